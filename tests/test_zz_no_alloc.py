"""fl_attn_decode_static: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc -- a serving loop that must not take the
device-wide synchronisation an allocation or a free can cause, or a plug-in
that does not own the process's device allocator -- and have no buffer to hand
over as a workspace.  fl_attn_decode_static serves them with the library's own
static scratch array (64 MiB).  Here it is called through the C ABI and
checked against fl_attn_decode (the same computation with a caller workspace)
and against the CPU oracle, on two calls in a row, since every call reuses the
array the previous one left behind; then a large multi-split call is followed
by a smaller one whose zero-initialised counters sit inside the larger call's
partial results; and a request larger than the array is refused with a clear
error.  This file is collected last, so a run that stops at its first failure
has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import attention_variant_gb300 as fa
import oracle
import testdata

torch = pytest.importorskip("torch")

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3  # the parity tolerances of every GPU test


def _paged_problem(tag, B, Sq, Hq, Hk, lens, page, seed):
    """A paged cache over a shuffled pool of pages (two spare pages), the
    device tensors for the library, and the same keys and values gathered
    into contiguous [B, S, Hk, 64] arrays for the oracle."""
    per = [-(-L // page) for L in lens]
    n_pages = sum(per) + 2
    perm = np.random.default_rng(seed).permutation(n_pages).astype(np.int32)
    table = np.full((B, max(per)), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, : per[b]] = perm[at: at + per[b]]
        at += per[b]
    q = testdata.normal_bf16((B, Sq, Hq, 64), tag, "q")
    kp = testdata.normal_bf16((n_pages, page, Hk, 64), tag, "k")
    vp = testdata.normal_bf16((n_pages, page, Hk, 64), tag, "v")
    S = max(per) * page
    k = np.zeros((B, S, Hk, 64), dtype=np.uint16)
    v = np.zeros((B, S, Hk, 64), dtype=np.uint16)
    for b in range(B):
        n = per[b] * page
        k[b, :n] = kp[table[b, : per[b]]].reshape(n, Hk, 64)
        v[b, :n] = vp[table[b, : per[b]]].reshape(n, Hk, 64)
    to = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    dev = dict(q=to(q), kp=to(kp), vp=to(vp),
               lens=torch.tensor(lens, dtype=torch.int32, device="cuda"),
               table=torch.from_numpy(table).cuda())
    return dev, (q, k, v)


def _small():
    return _paged_problem("no_alloc", 4, 2, 8, 2, (1100, 257, 129, 5), 64, 11)


def _large():
    lens = tuple(int(x) for x in np.random.default_rng(5).integers(3000, 8001, size=16))
    return _paged_problem("no_alloc_large", 16, 1, 32, 8, lens, 256, 12)


def _desc(dv, mod):
    return fa.make_decode_desc(dv["lens"], int(dv["lens"].max()), score_mod=mod, softcap=20.0,
                               causal=True, block_table=dv["table"])


def _static_call(dv, d):
    B, Sq, Hq, _ = dv["q"].shape
    out = torch.full((B, Sq, Hq, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    fa.fl_attn_decode_static(dv["q"], dv["kp"], dv["vp"], out, lse, d)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _check(o, lse, o_ref, lse_ref, what):
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, f"{what}: O differs by {err.max():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_MAX, f"{what}: LSE differs"


def _oracle(host, lens, mod):
    q, k, v = host
    return oracle.attention(q, k, v, mod=mod, softcap=20.0, mask="decode",
                            kv_len=np.asarray(lens, dtype=np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("mod", ["none", "softcap"])
def test_static_scratch_matches_workspace_call_twice(mod):
    dv, host = _small()
    B, Sq, Hq, _ = dv["q"].shape
    d = _desc(dv, mod)
    out_ref = torch.empty((B, Sq, Hq, 64), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fl_attn_decode_workspace_size(dv["q"], dv["kp"], d), dtype=torch.uint8,
                     device="cuda")
    fa.fl_attn_decode(dv["q"], dv["kp"], dv["vp"], out_ref, lse_ref, d, ws)
    torch.cuda.synchronize()
    o_ws, l_ws = out_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy()
    o_or, l_or = _oracle(host, dv["lens"].cpu().numpy(), mod)
    for call in range(2):
        o, l = _static_call(dv, d)
        _check(o, l, o_ws, l_ws, f"call {call} vs the workspace call")
        _check(o, l, o_or, l_or, f"call {call} vs the oracle")


@pytest.mark.gpu
def test_static_scratch_large_call_then_small_call():
    """A multi-split call over 16 long sequences fills far more of the array
    than the small problem needs; the small call that follows finds its
    counters inside those partial results and must still match the oracle."""
    big, big_host = _large()
    o, l = _static_call(big, _desc(big, "none"))
    _check(o, l, *_oracle(big_host, big["lens"].cpu().numpy(), "none"), "large call")
    dv, host = _small()
    o, l = _static_call(dv, _desc(dv, "none"))
    _check(o, l, *_oracle(host, dv["lens"].cpu().numpy(), "none"), "small call after the large one")


@pytest.mark.skipif(torch.cuda.is_available(), reason="made-up device addresses (host-only test)")
def test_static_scratch_refuses_oversize_requests():
    # 64 sequences x 64 KV heads x 4 splits (of 8 chunks of 128 keys) x 64 rows
    # x 64 fp32 = 256 MiB of partials, more than the 64 MiB array; refused
    # before any device work
    lib = fa.load_library()

    def t(shape):
        x = fa.FlTensor()
        x.ptr, x.dtype, x.ndim = 0x10000, fa.FL_BF16, len(shape)
        acc = 1
        for dim in range(len(shape) - 1, -1, -1):
            x.sizes[dim] = shape[dim]
            x.strides[dim] = acc
            acc *= shape[dim]
        return x

    d = fa.FlDecodeDesc()
    d.kv_lens = 0x20000
    d.max_kv_len = 4096
    d.causal = 1
    q, kc, o = t((64, 1, 4096, 64)), t((64, 4096, 64, 64)), t((64, 1, 4096, 64))
    st = lib.fl_attn_decode_static(ctypes.byref(q), ctypes.byref(kc), ctypes.byref(kc),
                                   ctypes.byref(o), None, ctypes.byref(d), None)
    assert st == fa.FL_ERR_UNSUPPORTED
    assert "static decode scratch holds" in fa.fl_attn_last_error()
