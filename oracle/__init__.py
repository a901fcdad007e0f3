"""CPU oracle for the fused attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library neither imports it nor shares
any code with it; ``fl_oracle.c`` is compiled on its own by :func:`build`.

Every function returns float64 results for the bf16 inputs it is given (as
uint16 bit patterns).  The definitions followed are those of the Flashlight
pages: an attention forward ``softmax(score_mod(scale QK^T) + mask + bias) V``
whose online-softmax rewrite is exact over the reals (gist.science summary,
"Methodology" item 3; talk notes, "Compiler design 2: algebraic
transformation").  The variant formulas come from the workload statement that
accompanies the pages; ``fl_oracle.c`` lists them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fl_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libfloracle.so")

MOD = {"none": 0, "alibi": 1, "softcap": 2}
MASK = {"none": 0, "causal": 1, "window": 2, "prefix": 3, "doc": 4, "kv_len": 5, "decode": 6}


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hk", ctypes.c_int32),
        ("Sq", ctypes.c_int32), ("Sk", ctypes.c_int32), ("D", ctypes.c_int32),
        ("Dv", ctypes.c_int32),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3),
        ("score_mod", ctypes.c_int32), ("softcap", ctypes.c_double),
        ("alibi_slopes", ctypes.c_void_p),
        ("mask", ctypes.c_int32), ("window", ctypes.c_int32), ("prefix", ctypes.c_int32),
        ("doc_offsets", ctypes.c_void_p), ("doc_stride", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("bias", ctypes.c_void_p), ("bias_stride", ctypes.c_int64 * 3),
        ("kv_len", ctypes.c_void_p),
        ("key_mask", ctypes.c_void_p), ("key_mask_stride", ctypes.c_int64 * 2),
    ]


def build(force: bool = False, source: str = _SRC, target: str = _LIB) -> str:
    """Compile ``fl_oracle.c`` into a shared library (plain C11 + OpenMP)."""
    os.makedirs(os.path.dirname(target), exist_ok=True)
    if (not force and os.path.exists(target)
            and os.path.getmtime(target) >= os.path.getmtime(source)):
        return target
    tmp = target + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


_lib = None


def load(path: str | None = None):
    """Load (building if needed) the oracle library."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
    lib.fl_oracle_attention.restype = ctypes.c_int
    lib.fl_oracle_attention.argtypes = [
        ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.fl_oracle_max_threads.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def max_threads() -> int:
    return int(load().fl_oracle_max_threads())


def _bshd_strides(a: np.ndarray) -> tuple[int, int, int]:
    """Element strides of axes (batch, position, head) of a [B, S, H, D] view."""
    if a.dtype != np.uint16 or a.ndim != 4 or a.strides[3] != 2:
        raise ValueError("expected a [B, S, H, D] uint16 view with contiguous features")
    return tuple(s // 2 for s in a.strides[:3])


def _base_and_span(a: np.ndarray):
    """Pointer to element 0 of a possibly-strided view."""
    return a.__array_interface__["data"][0]


def attention(q, k, v, *, mod="none", softcap=20.0, alibi_slopes=None, mask="none",
              window=0, prefix=0, doc_offsets=None, scale=0.0, bias=None, kv_len=None,
              key_mask=None, rows=None, nthreads=0, lib=None):
    """Attention forward of ``q [B,Sq,Hq,D]``, ``k [B,Sk,Hk,D]``, ``v [B,Sk,Hk,Dv]``.

    ``bias`` (optional) is ``[Hq, Sq, Sk]`` bf16 bits.  ``doc_offsets`` is the
    int32 ``[B, max_docs+1]`` table of document starts padded with ``Sk``.
    ``kv_len`` (masks ``kv_len`` and ``decode``) holds each batch element's
    cache length; the decode mask puts the ``Sq`` query rows at the last
    ``Sq`` positions of that length.
    ``key_mask`` (optional, ``[B, Sk]``) removes key j of batch element b
    where it is zero, on top of ``mask``.
    ``rows`` (optional) is an ``[n, 3]`` array of ``(b, h, i)``; then the
    result is ``O [n, Dv]`` and ``LSE [n]``, else ``O [B,Sq,Hq,Dv]`` and
    ``LSE [B,Hq,Sq]``.
    """
    lib = lib or load()
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hk, Dk = k.shape
    Dv = v.shape[3]
    if Bk != B or Dk != D or v.shape[:3] != (B, Sk, Hk) or Hq % Hk:
        raise ValueError("inconsistent shapes")
    p = _Problem()
    p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.D, p.Dv = B, Hq, Hk, Sq, Sk, D, Dv
    p.q_stride[:] = _bshd_strides(q)
    p.k_stride[:] = _bshd_strides(k)
    p.v_stride[:] = _bshd_strides(v)
    p.score_mod = MOD[mod]
    p.softcap = float(softcap)
    keep = []
    if alibi_slopes is not None:
        sl = np.ascontiguousarray(alibi_slopes, dtype=np.float64)
        keep.append(sl)
        p.alibi_slopes = sl.ctypes.data
    p.mask = MASK[mask]
    p.window = int(window)
    p.prefix = int(prefix)
    if doc_offsets is not None:
        do = np.ascontiguousarray(doc_offsets, dtype=np.int32)
        keep.append(do)
        p.doc_offsets = do.ctypes.data
        p.doc_stride = do.shape[1]
    p.scale = float(scale)
    if kv_len is not None:
        kl = np.ascontiguousarray(kv_len, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("kv_len must have one entry per batch element")
        keep.append(kl)
        p.kv_len = kl.ctypes.data
    if key_mask is not None:
        km = np.ascontiguousarray(np.asarray(key_mask) != 0, dtype=np.uint8)
        if km.shape != (B, Sk):
            raise ValueError("key_mask must be [B, Sk]")
        keep.append(km)
        p.key_mask = km.ctypes.data
        p.key_mask_stride[:] = (Sk, 1)
    if bias is not None:
        if bias.dtype != np.uint16 or bias.shape != (Hq, Sq, Sk):
            raise ValueError("bias must be [Hq, Sq, Sk] bf16 bits")
        p.bias = _base_and_span(bias)
        p.bias_stride[:] = tuple(s // 2 for s in bias.strides)
    if rows is None:
        out = np.zeros((B, Sq, Hq, Dv), dtype=np.float64)
        lse = np.zeros((B, Hq, Sq), dtype=np.float64)
        rp, n = None, 0
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        keep.append(r)
        out = np.zeros((r.shape[0], Dv), dtype=np.float64)
        lse = np.zeros((r.shape[0],), dtype=np.float64)
        rp, n = r.ctypes.data, r.shape[0]
    rc = lib.fl_oracle_attention(ctypes.byref(p), _base_and_span(q), _base_and_span(k),
                                 _base_and_span(v), rp, n, out.ctypes.data,
                                 lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle rejected the problem")
    return out, lse


def diff_attention(q, k, v, lam, *, mask="none", scale=0.0, rows=None, nthreads=0, lib=None):
    """Differential attention: ``(softmax(Q1 K1^T s) - lam softmax(Q2 K2^T s)) V``.

    ``q [2,B,S,H,D]``, ``k [2,B,S,Hk,D]``, ``v [B,S,Hk,Dv]``.  Two independent
    softmaxes (each with its own max and sum), one shared V (the pages name
    differential attention among the complex variants: gist.science summary,
    "Results"; the formula is the workload statement's).  Returns O and the
    per-stream LSE stacked on a leading axis of 2.
    """
    o1, l1 = attention(q[0], k[0], v, mask=mask, scale=scale, rows=rows, nthreads=nthreads,
                       lib=lib)
    o2, l2 = attention(q[1], k[1], v, mask=mask, scale=scale, rows=rows, nthreads=nthreads,
                       lib=lib)
    return o1 - lam * o2, np.stack([l1, l2])


def sigmoid_bf16(g):
    """sigmoid of bf16 bit patterns, in float64."""
    x = (np.asarray(g, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return 1.0 / (1.0 + np.exp(-x.astype(np.float64)))


def evo_row(q, k, v, bias, gate, *, msa_mask=None, rows=None, nthreads=0, lib=None):
    """Evoformer row-wise gated self-attention with pair bias.

    ``q, k, v, gate`` are ``[N_seq, N_res, H, c]``; ``bias`` is
    ``[H, N_res, N_res]`` shared by every MSA row.  For each MSA row s and head
    h, attention runs over residues with ``b[h, i, j]`` added to the logits;
    the output is gated by ``sigmoid(g[s, i, h, :])`` (talk notes, "End-to-end:
    AlphaFold2"; shapes from the workload statement).  ``msa_mask``
    (optional, ``[N_seq, N_res]``) removes residue j as a key of MSA row s
    where it is zero.  With ``rows`` the triples are ``(s, h, i)``.
    """
    o, lse = attention(q, k, v, bias=bias, key_mask=msa_mask, rows=rows, nthreads=nthreads,
                       lib=lib)
    if rows is None:
        o = o * sigmoid_bf16(gate)
    else:
        r = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
        o = o * sigmoid_bf16(gate[r[:, 0], r[:, 2], r[:, 1], :])
    return o, lse


def evo_col(q, k, v, gate, *, msa_mask=None, rows=None, nthreads=0, lib=None):
    """Evoformer column-wise gated self-attention (no bias).

    Attention for each residue r and head h runs over the MSA rows (axis 0) of
    the same ``[N_seq, N_res, H, c]`` tensors; the gate is the same
    ``sigmoid(g[s, r, h, :])``.  ``msa_mask`` (optional, ``[N_seq, N_res]``)
    removes MSA row t as a key of residue r where ``msa_mask[t, r]`` is zero.
    Results are laid out ``O [N_res, N_seq, H, c]`` and ``LSE [N_res, H, N_seq]``;
    with ``rows`` the triples are ``(r, h, s)``.
    """
    qt, kt, vt = (np.swapaxes(x, 0, 1) for x in (q, k, v))
    km = None if msa_mask is None else np.swapaxes(np.asarray(msa_mask), 0, 1)
    o, lse = attention(qt, kt, vt, key_mask=km, rows=rows, nthreads=nthreads, lib=lib)
    gt = np.swapaxes(gate, 0, 1)
    if rows is None:
        o = o * sigmoid_bf16(gt)
    else:
        r = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
        o = o * sigmoid_bf16(gt[r[:, 0], r[:, 2], r[:, 1], :])
    return o, lse


def alibi_slopes(H: int) -> np.ndarray:
    """``slope_h = 2^(-8 (h+1) / H)`` for 0-based h (workload statement)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=np.float64)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))


def _allowed(mask, S, b, window, prefix, doc_offsets):
    """Boolean [S, S] matrix of allowed (query i, key j) pairs, from the mask
    predicates (the same definitions fl_oracle.c states)."""
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if mask == "none":
        return np.ones((S, S), dtype=bool)
    if mask == "causal":
        return j <= i
    if mask == "window":
        return (j <= i) & (i - j < window)
    if mask == "prefix":
        return (j <= i) | (j < prefix)
    if mask == "doc":
        starts = np.asarray(doc_offsets)[b]
        doc = np.searchsorted(starts, np.arange(S), side="right") - 1  # starts <= x, minus one
        return (j <= i) & (doc[:, None] == doc[None, :])
    raise ValueError(mask)


def attention_bwd(q, k, v, dout, *, mod="none", softcap=20.0, alibi_slopes=None, expr=None, mask="none",
                  window=0, prefix=0, doc_offsets=None, scale=0.0):
    """Gradients dQ, dK, dV (float64) of ``O = softmax(scale Q K^T + mask) V``
    for ``q [B,S,Hq,D]``, ``k, v [B,S,Hk,D]`` and the output gradient
    ``dout [B,S,Hq,D]`` (all bf16 bits), with any mask of ``attention``
    (none, causal, window, prefix, doc) and score_mod none, ALiBi or softcap:
    z = score_mod(u), u = scale q.k, and the chain rule takes dL/dz to dL/du
    (1 for ALiBi, an additive bias; 1 - tanh^2(u / cap) for softcap; for
    ``mod="expr"`` the derivative of the score_mod expression ``expr``, from
    :func:`oracle.score_expr.evaluate_with_grad`).

    The plain definition per (batch, query head): the full probability matrix
    P (two-pass softmax), dV = P^T dO, dP = dO V^T, dS_ij = P_ij (dP_ij -
    sum_l P_il dP_il), dQ = scale dS K, dK = scale dS^T Q; query heads sharing
    a K/V head add their dK and dV (gist.science summary, "Limitations and
    future work": the backward pass is the fused kernels' next step).
    """
    wid = lambda x: (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32) \
        .astype(np.float64)
    Q, K, V, dO = wid(q), wid(k), wid(v), wid(dout)
    B, S, Hq, D = Q.shape
    Hk = K.shape[2]
    G = Hq // Hk
    s = scale if scale else 1.0 / np.sqrt(D)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    slopes = alibi_slopes if alibi_slopes is not None else globals()["alibi_slopes"](Hq)
    dist = np.abs(np.arange(S)[:, None] - np.arange(S)[None, :]).astype(np.float64)
    for b in range(B):
        allowed = _allowed(mask, S, b, window, prefix, doc_offsets)
        for h in range(Hq):
            kh = h // G
            u = s * (Q[b, :, h] @ K[b, :, kh].T)
            chain = 1.0
            if mod == "alibi":
                z = u - slopes[h] * dist
            elif mod == "softcap":
                th = np.tanh(u / softcap)
                z = softcap * th
                chain = 1.0 - th * th
            elif mod == "expr":
                from oracle import score_expr
                z, chain = score_expr.evaluate_with_grad(
                    expr, score=u, b=float(b), h=float(h), q_idx=np.arange(S, dtype=np.float64)[:, None],
                    kv_idx=np.arange(S, dtype=np.float64)[None, :])
                z, chain = np.broadcast_to(z, u.shape), np.broadcast_to(chain, u.shape)
            else:
                z = u
            z = np.where(allowed, z, -np.inf)
            m = z.max(axis=1, keepdims=True)
            e = np.exp(z - m)
            P = e / e.sum(axis=1, keepdims=True)
            dV[b, :, kh] += P.T @ dO[b, :, h]
            dP = dO[b, :, h] @ V[b, :, kh].T
            with np.errstate(invalid="ignore"):
                dS = np.where(P > 0, P * (dP - (P * dP).sum(axis=1, keepdims=True)) * chain, 0.0)
            dQ[b, :, h] = s * (dS @ K[b, :, kh])
            dK[b, :, kh] += s * (dS.T @ Q[b, :, h])
    return dQ, dK, dV


def diff_attention_bwd(q, k, v, dout, lam, *, mask="none", scale=0.0):
    """Gradients of differential attention, float64:
    ``O = softmax(s Q1 K1^T + mask) V - lam softmax(s Q2 K2^T + mask) V``
    for ``q [2,B,S,H,D]``, ``k [2,B,S,Hk,D]``, ``v [B,S,Hk,Dv]`` and
    ``dout [B,S,H,Dv]`` (bf16 bits); returns ``dQ [2,B,S,H,D]``,
    ``dK [2,B,S,Hk,D]``, ``dV [B,S,Hk,Dv]``.

    The chain rule through both softmaxes, written out per (batch, head):
    stream t has its own probability matrix P_t and the coefficient c_t
    (1, then -lam) on its output, so dP_t = c_t dO V^T, dS_t = P_t (dP_t -
    rowsum(P_t dP_t)), dQ_t = s dS_t K_t, dK_t = s dS_t^T Q_t, and the shared
    V collects dV = sum_t c_t P_t^T dO.  (Differential attention is one of
    the pages' complex variants, gist.science summary, "Results"; the backward
    is the fused kernels' named next step, "Limitations and future work".)
    """
    wid = lambda x: (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32) \
        .astype(np.float64)
    Q, K, V, dO = wid(q), wid(k), wid(v), wid(dout)
    _, B, S, H, D = Q.shape
    Hk = K.shape[3]
    G = H // Hk
    sc = scale if scale else 1.0 / np.sqrt(D)
    coef = (1.0, -float(lam))
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for b in range(B):
        allowed = _allowed(mask, S, b, 0, 0, None)
        for h in range(H):
            kh = h // G
            for t in range(2):
                z = np.where(allowed, sc * (Q[t, b, :, h] @ K[t, b, :, kh].T), -np.inf)
                e = np.exp(z - z.max(axis=1, keepdims=True))
                P = e / e.sum(axis=1, keepdims=True)
                dV[b, :, kh] += coef[t] * (P.T @ dO[b, :, h])
                dP = coef[t] * (dO[b, :, h] @ V[b, :, kh].T)
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dQ[t, b, :, h] = sc * (dS @ K[t, b, :, kh])
                dK[t, b, :, kh] += sc * (dS.T @ Q[t, b, :, h])
    return dQ, dK, dV
