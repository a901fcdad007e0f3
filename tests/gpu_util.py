"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
on seeded inputs and compare with the oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import attention_variant_gb300 as fa

# Tolerances of the parity bar: O with bf16 inputs and fp32 accumulation,
# max |err| <= 1e-2 and mean |err| <= 1e-3; LSE max |err| <= 1e-3.
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3


def dev(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns -> bf16 CUDA tensor with the same bytes."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_standard(q, k, v, *, lse=True, counts=True, layout="bshd", **desc):
    """q/k/v: bf16-bit numpy [B,S,H,D].  Returns (O f64, LSE f64 or None,
    tile counts or None, error word)."""
    B, S, Hq, D = q.shape
    Hk, Dv = k.shape[2], v.shape[3]
    if layout == "bhsd":  # store B,H,S,D and pass a strided BSHD view
        qd, kd, vd = (dev(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
                      for x in (q, k, v))
        out = torch.empty((B, Hq, S, Dv), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    else:
        qd, kd, vd = dev(q), dev(k), dev(v)
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device="cuda")
    out.fill_(float("nan"))
    lse_t = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    nq = (S + 127) // 128
    cnt = torch.full((B, Hq, nq), -1, dtype=torch.int32, device="cuda") if counts else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    doc = desc.pop("doc_offsets", None)
    doc_t = torch.from_numpy(np.ascontiguousarray(doc, dtype=np.int32)).cuda() if doc is not None else None
    d = fa.make_desc(doc_offsets=doc_t, debug_tile_counts=cnt, error_word=err, **desc)
    fa.fl_attn_fwd(qd, kd, vd, out, lse_t, d)
    torch.cuda.synchronize()
    return (f64(out), f64(lse_t) if lse else None,
            cnt.cpu().numpy() if counts else None, int(err.item()))


def compare(o, lse, o_ref, lse_ref, what=""):
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert err.max() <= O_MAX, f"{what}: O max err {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: O mean err {err.mean():.3e}"
    if lse is not None:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin), f"{what}: LSE finiteness differs"
        if fin.any():
            e = np.abs(lse[fin] - lse_ref[fin]).max()
            assert e <= LSE_MAX, f"{what}: LSE max err {e:.3e}"
    return float(err.max()), float(err.mean())


def row_interval(mask, i, S, window=0, prefix=0, starts=None):
    """Allowed keys [lo, hi) of query row i, from each mask's definition."""
    if mask == "none":
        return 0, S
    if mask == "causal":
        return 0, min(i + 1, S)
    if mask == "window":
        return max(0, i - window + 1), min(i + 1, S)
    if mask == "prefix":
        return 0, min(S, max(i + 1, prefix))
    if mask == "doc":
        return int(starts[starts <= i].max()), min(i + 1, S)
    raise ValueError(mask)


def expected_tile_counts(mask, B, H, S, window=0, prefix=0, doc=None, bm=128, bn=128):
    """Visited KV tiles per (b, h, query block): ceil(hi / bn) - floor(lo / bn)
    over the union [lo, hi) of the block's allowed keys (computed here by
    brute force over the rows of each block)."""
    nq = (S + bm - 1) // bm
    out = np.zeros((B, H, nq), dtype=np.int64)
    for b in range(B):
        starts = None if doc is None else np.asarray(doc[b])
        for qb in range(nq):
            rows = range(qb * bm, min(qb * bm + bm, S))
            ivs = [row_interval(mask, i, S, window, prefix, starts) for i in rows]
            lo = min(a for a, _ in ivs)
            hi = max(z for _, z in ivs)
            out[b, :, qb] = -(-hi // bn) - lo // bn
    return out


def sample_rows(B, H, S, n, seed=0):
    """Seeded (b, h, i) triples that always include the first and last rows
    and the tile edges."""
    rng = np.random.default_rng(seed)
    fixed = [0, S - 1, min(127, S - 1), min(128, S - 1), S // 2]
    rows = []
    for t in range(n):
        i = fixed[t] if t < len(fixed) else int(rng.integers(0, S))
        rows.append((int(rng.integers(0, B)), int(rng.integers(0, H)), i))
    return np.array(rows, dtype=np.int64)


def block_edge_rows(B, H, S, n_random=0, seed=0, bm=128):
    """(b, h, i) triples: the first and the last query row of every
    (batch, head, 128-row query block), plus `n_random` seeded rows."""
    rows = []
    for b in range(B):
        for h in range(H):
            for q0 in range(0, S, bm):
                rows.append((b, h, q0))
                last = min(q0 + bm, S) - 1
                if last != q0:
                    rows.append((b, h, last))
    rng = np.random.default_rng(seed)
    for _ in range(n_random):
        rows.append((int(rng.integers(0, B)), int(rng.integers(0, H)), int(rng.integers(0, S))))
    return np.array(rows, dtype=np.int64)
