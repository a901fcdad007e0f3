"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or a
deliberately broken copy built by ``test_oracle_mutants.py``) and raises
``AssertionError`` when the oracle disagrees with

* a closed form (constant scores give the mean of V over the allowed keys and
  LSE = ln(#allowed); ALiBi over constant scores is a geometric series; a
  two-key softcap problem; the Evoformer gate and the differential lambda on
  constant scores),
* an invariant (rows of P sum to one; per-row shift of the logits leaves O
  unchanged and moves LSE by the shift; non-causal attention is equivariant
  under a joint permutation of keys and values; causal row 0 returns v_0),
* a library routine (float64 ``torch.nn.functional.scaled_dot_product_attention``
  for vanilla, causal, boolean masks, ALiBi as an additive mask and GQA), or
* a special case that reduces to another variant.

None of these restates the oracle's row loop.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import testdata

ATOL = 1e-10


def _bf(x) -> np.ndarray:
    """float array -> bf16 bit patterns (values chosen exactly representable)."""
    bits = testdata.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    back = testdata.bf16_bits_to_f32(bits)
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "value not exact in bf16"
    return bits


def _f64(bits) -> np.ndarray:
    return testdata.bf16_bits_to_f32(bits).astype(np.float64)


def _rand(shape, name, wl="pins"):
    return testdata.normal_bf16(shape, wl, name)


def _sdpa(q, k, v, mask=None, enable_gqa=False, scale=None):
    """float64 SDPA over [B,S,H,D] bf16-bit inputs; returns O [B,S,H,Dv]."""
    Q, K, V = (torch.from_numpy(_f64(x)).permute(0, 2, 1, 3) for x in (q, k, v))
    kw = {}
    if enable_gqa:
        kw["enable_gqa"] = True
    if scale is not None:
        kw["scale"] = scale
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, **kw)
    return o.permute(0, 2, 1, 3).numpy()


def _close(a, b, atol=ATOL, what=""):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= atol, f"{what}: max |err| {err:.3e} > {atol:.1e}"


# --------------------------------------------------------------------------
# closed forms on constant scores (Q = 0)


def _allowed_range(mask, i, S, window=0, prefix=0, starts=None):
    """[lo, hi) of keys allowed for row i, from the interval form of each mask."""
    if mask == "none":
        return 0, S
    if mask == "causal":
        return 0, i + 1
    if mask == "window":
        return max(0, i - window + 1), i + 1
    if mask == "prefix":
        return 0, max(i + 1, min(prefix, S))
    if mask == "doc":
        ds = max(s for s in starts if s <= i)
        return ds, i + 1
    raise ValueError(mask)


def pin_constant_scores(lib):
    """Q = 0: every allowed key has logit 0, so O_i = mean of V over the
    allowed keys (via prefix sums) and LSE_i = ln(number allowed)."""
    S, H, D, Dv = 300, 2, 64, 64
    q = _bf(np.zeros((2, S, H, D)))
    k = _rand((2, S, H, D), "k")
    v = _rand((2, S, H, Dv), "v")
    vf = _f64(v)
    csum = np.concatenate([np.zeros((2, 1, H, Dv)), np.cumsum(vf, axis=1)], axis=1)
    starts = [[0, 37, 38, 120, 260], [0, 150]]
    doc = np.full((2, 6), S, dtype=np.int32)
    for b, st in enumerate(starts):
        doc[b, : len(st)] = st
    for mask, kw in [("none", {}), ("causal", {}), ("window", {"window": 37}),
                     ("prefix", {"prefix": 50}), ("doc", {"doc_offsets": doc})]:
        o, lse = oracle.attention(q, k, v, mask=mask, lib=lib, **kw)
        for b in range(2):
            for i in range(S):
                lo, hi = _allowed_range(mask, i, S, kw.get("window", 0), kw.get("prefix", 0),
                                        starts[b] if mask == "doc" else None)
                mean = (csum[b, hi] - csum[b, lo]) / (hi - lo)
                _close(o[b, i], mean, what=f"{mask} O row {i}")
                _close(lse[b, :, i], math.log(hi - lo), what=f"{mask} LSE row {i}")


def pin_alibi_geometric(lib):
    """Q = 0 with ALiBi and no mask: z_ij = -slope_h |i-j|, so with r = e^-slope
    LSE_i = ln(1 + r(1-r^i)/(1-r) + r(1-r^(S-1-i))/(1-r)), and with V = 1 the
    output is 1.  Default slopes must be 2^(-8(h+1)/H)."""
    S, H, D = 40, 4, 64
    q = _bf(np.zeros((1, S, H, D)))
    k = _rand((1, S, H, D), "k")
    v = _bf(np.ones((1, S, H, 8)))
    o, lse = oracle.attention(q, k, v, mod="alibi", lib=lib)
    _close(o, 1.0, what="alibi P row sums")
    for h in range(H):
        r = math.exp(-(2.0 ** (-8.0 * (h + 1) / H)))
        for i in range(S):
            left = r * (1 - r ** i) / (1 - r)
            right = r * (1 - r ** (S - 1 - i)) / (1 - r)
            _close(lse[0, h, i], math.log(1 + left + right), what=f"alibi LSE h{h} i{i}")
    # O with V = position index: the weighted mean of j under the geometric weights
    vpos = _bf(np.broadcast_to(np.arange(S, dtype=np.float32)[None, :, None, None],
                               (1, S, H, 8)).copy())
    o, _ = oracle.attention(q, k, vpos, mod="alibi", lib=lib)
    for h in (0, H - 1):
        r = math.exp(-(2.0 ** (-8.0 * (h + 1) / H)))
        for i in (0, 7, S - 1):
            w = np.array([r ** abs(i - j) for j in range(S)])
            _close(o[0, i, h, 0], float(np.dot(w, np.arange(S)) / w.sum()),
                   what=f"alibi mean position h{h} i{i}")


def pin_softcap_two_keys(lib):
    """Two keys with scores a and 0 (q = x e_0, k_0 = y e_0, k_1 = 0): the
    logits are cap*tanh(a/cap) and 0, so LSE = ln(1 + e^(cap tanh(a/cap)))
    and O = sigmoid(cap tanh(a/cap)) v_0 + (1 - sigmoid) v_1."""
    D, cap = 64, 20.0
    for x, y in [(8.0, 4.0), (32.0, 24.0), (-16.0, 12.0), (64.0, 64.0)]:
        q = np.zeros((1, 1, 1, D)); q[..., 0] = x
        k = np.zeros((1, 2, 1, D)); k[0, 0, 0, 0] = y
        v = np.zeros((1, 2, 1, 2)); v[0, 0, 0] = (1.0, 0.0); v[0, 1, 0] = (0.0, 1.0)
        o, lse = oracle.attention(_bf(q), _bf(k), _bf(v), mod="softcap", softcap=cap, lib=lib)
        a = x * y / math.sqrt(D)
        z = cap * math.tanh(a / cap)
        _close(lse[0, 0, 0], math.log1p(math.exp(z)), what=f"softcap LSE a={a}")
        sg = 1.0 / (1.0 + math.exp(-z))
        _close(o[0, 0, 0], [sg, 1 - sg], what=f"softcap O a={a}")


def pin_one_hot(lib):
    """q_i = c e_t and only key j* carries e_t: with c large the softmax is
    one-hot and O_i = v_{j*} exactly; logits near 1000 also require the max
    to be subtracted before exponentiating."""
    S, D = 16, 64
    c = 8000.0
    q = np.zeros((1, S, 1, D)); q[..., 5] = c
    k = np.zeros((1, S, 1, D)); k[0, 11, 0, 5] = 1.0
    v = _rand((1, S, 1, D), "v1")
    o, lse = oracle.attention(_bf(q), _bf(k), v, lib=lib)
    for i in range(S):
        _close(o[0, i, 0], _f64(v)[0, 11, 0], what="one-hot O")
        _close(lse[0, 0, i], c / 8.0, atol=1e-9, what="one-hot LSE")


def pin_rows_sum_to_one(lib):
    """V = 1 gives O = sum_j P_ij = 1 for every variant and mask."""
    S, H = 130, 2
    q, k = _rand((1, S, H, 64), "q2"), _rand((1, S, H, 64), "k2")
    v = _bf(np.ones((1, S, H, 4)))
    doc = np.array([[0, 64, 100, S]], dtype=np.int32)
    for mod in ("none", "alibi", "softcap"):
        for mask, kw in [("none", {}), ("causal", {}), ("window", {"window": 9}),
                         ("prefix", {"prefix": 33}), ("doc", {"doc_offsets": doc})]:
            o, _ = oracle.attention(q, k, v, mod=mod, mask=mask, lib=lib, **kw)
            _close(o, 1.0, atol=1e-12, what=f"{mod}/{mask} row sums")


def pin_shift_invariance(lib):
    """A bias constant along each row (b[h,i,j] = c_{h,i}) leaves O unchanged
    and shifts LSE by c_{h,i}; a transposed bias index would break both."""
    S, H = 48, 2
    q, k, v = (_rand((1, S, H, 64), n) for n in ("q3", "k3", "v3"))
    c = np.array([[(-1) ** i * (i % 7) * 0.5 for i in range(S)] for _ in range(H)])
    bias = _bf(np.broadcast_to(c[:, :, None], (H, S, S)).copy())
    o0, l0 = oracle.attention(q, k, v, lib=lib)
    o1, l1 = oracle.attention(q, k, v, bias=bias, lib=lib)
    _close(o1, o0, atol=1e-12, what="shift O")
    _close(l1[0], l0[0] + c, atol=1e-12, what="shift LSE")


def pin_permutation(lib):
    """Non-causal vanilla: permuting keys and values together leaves O and LSE
    unchanged; permuting queries permutes the outputs."""
    S, H = 77, 2
    q, k, v = (_rand((1, S, H, 64), n) for n in ("q4", "k4", "v4"))
    perm = np.random.default_rng(7).permutation(S)
    o0, l0 = oracle.attention(q, k, v, lib=lib)
    o1, l1 = oracle.attention(q, np.ascontiguousarray(k[:, perm]),
                              np.ascontiguousarray(v[:, perm]), lib=lib)
    _close(o1, o0, atol=1e-12, what="KV permutation O")
    _close(l1, l0, atol=1e-12, what="KV permutation LSE")
    o2, _ = oracle.attention(np.ascontiguousarray(q[:, perm]), k, v, lib=lib)
    _close(o2, o0[:, perm], atol=1e-12, what="Q permutation")


def pin_causal_row0(lib):
    """Causal row 0 sees only key 0: O_0 = v_0 and LSE_0 = scale q_0 . k_0."""
    S, H = 20, 2
    q, k, v = (_rand((2, S, H, 64), n) for n in ("q5", "k5", "v5"))
    o, lse = oracle.attention(q, k, v, mask="causal", lib=lib)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    _close(o[:, 0], vf[:, 0], what="causal row 0 O")
    z00 = np.einsum("bhd,bhd->bh", qf[:, 0], kf[:, 0]) / 8.0
    _close(lse[:, :, 0], z00, what="causal row 0 LSE")


def pin_sdpa(lib):
    """float64 SDPA agreement: vanilla, causal, every mask as a boolean
    attn_mask built by broadcast index comparisons, ALiBi as an additive
    mask, GQA with enable_gqa, a custom scale and a strided (BHSD) layout."""
    B, S, H, D = 2, 70, 4, 64
    q, k, v = (_rand((B, S, H, D), n) for n in ("q6", "k6", "v6"))
    o, _ = oracle.attention(q, k, v, lib=lib)
    _close(o, _sdpa(q, k, v), what="SDPA vanilla")
    o, _ = oracle.attention(q, k, v, scale=0.05, lib=lib)
    _close(o, _sdpa(q, k, v, scale=0.05), what="SDPA scale")
    ii = np.arange(S)[:, None]
    jj = np.arange(S)[None, :]
    doc = np.array([[0, 13, 14, 50, S], [0, 40, S, S, S]], dtype=np.int32)
    docid = np.stack([np.searchsorted(doc[b], np.arange(S), side="right") - 1 for b in range(B)])
    masks = {
        "causal": ({}, np.broadcast_to(jj <= ii, (B, 1, S, S))),
        "window": ({"window": 11}, np.broadcast_to((jj <= ii) & (ii - jj < 11), (B, 1, S, S))),
        "prefix": ({"prefix": 23}, np.broadcast_to((jj <= ii) | (jj < 23), (B, 1, S, S))),
        "doc": ({"doc_offsets": doc},
                (docid[:, None, :, None] == docid[:, None, None, :]) & (jj <= ii)[None, None]),
    }
    for name, (kw, m) in masks.items():
        o, _ = oracle.attention(q, k, v, mask=name, lib=lib, **kw)
        _close(o, _sdpa(q, k, v, mask=torch.from_numpy(np.ascontiguousarray(m))),
               what=f"SDPA {name}")
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])
    add = torch.from_numpy(-slopes[None, :, None, None] * np.abs(ii - jj)[None, None])
    o, _ = oracle.attention(q, k, v, mod="alibi", lib=lib)
    _close(o, _sdpa(q, k, v, mask=add), what="SDPA alibi")
    Hk = 2
    k2, v2 = _rand((B, S, Hk, D), "k7"), _rand((B, S, Hk, D), "v7")
    o, _ = oracle.attention(q, k2, v2, lib=lib)
    _close(o, _sdpa(q, k2, v2, enable_gqa=True), what="SDPA GQA")
    o, _ = oracle.attention(q, k2, v2, mask="causal", lib=lib)
    _close(o, _sdpa(q, k2, v2, mask=torch.from_numpy(np.ascontiguousarray(
        np.broadcast_to(jj <= ii, (B, 1, S, S)))), enable_gqa=True), what="SDPA GQA causal")
    # BHSD storage passed as a strided BSHD view
    qh = np.ascontiguousarray(q.transpose(0, 2, 1, 3)).transpose(0, 2, 1, 3)
    o, _ = oracle.attention(qh, k, v, lib=lib)
    _close(o, _sdpa(q, k, v), what="SDPA strided")


def pin_reductions(lib):
    """Special cases that reduce to another variant."""
    S, H = 90, 2
    q, k, v = (_rand((1, S, H, 64), n) for n in ("q8", "k8", "v8"))
    van = oracle.attention(q, k, v, lib=lib)
    cau = oracle.attention(q, k, v, mask="causal", lib=lib)
    pairs = [
        (oracle.attention(q, k, v, mod="softcap", softcap=1e30, lib=lib), van, "softcap inf"),
        (oracle.attention(q, k, v, mod="alibi", alibi_slopes=np.zeros(H), lib=lib), van,
         "alibi 0"),
        (oracle.attention(q, k, v, mask="window", window=S, lib=lib), cau, "window S"),
        (oracle.attention(q, k, v, mask="prefix", prefix=0, lib=lib), cau, "prefix 0"),
        (oracle.attention(q, k, v, mask="prefix", prefix=S, lib=lib), van, "prefix S"),
        (oracle.attention(q, k, v, mask="doc", doc_offsets=np.array([[0, S]], np.int32),
                          lib=lib), cau, "one document"),
    ]
    for (o1, l1), (o0, l0), what in pairs:
        _close(o1, o0, atol=1e-12, what=what)
        _close(l1, l0, atol=1e-9, what=what + " LSE")
    # GQA equals MHA on repeat-interleaved K/V
    k2, v2 = _rand((1, S, 1, 64), "k9"), _rand((1, S, 1, 64), "v9")
    o1, _ = oracle.attention(q, k2, v2, mask="causal", lib=lib)
    o0, _ = oracle.attention(q, np.repeat(k2, H, axis=2), np.repeat(v2, H, axis=2),
                             mask="causal", lib=lib)
    _close(o1, o0, atol=1e-12, what="GQA repeat")


def pin_rows_api(lib):
    """Sampled rows equal the same rows of the full result."""
    S, H = 140, 4
    q, k = _rand((2, S, H, 64), "qa"), _rand((2, S, 2, 64), "ka")
    v = _rand((2, S, 2, 32), "va")
    o, lse = oracle.attention(q, k, v, mask="window", window=50, mod="alibi", lib=lib)
    rows = np.array([[0, 0, 0], [1, 3, 139], [0, 2, 77], [1, 1, 5]])
    o2, l2 = oracle.attention(q, k, v, mask="window", window=50, mod="alibi", rows=rows, lib=lib)
    for n, (b, h, i) in enumerate(rows):
        _close(o2[n], o[b, i, h], atol=0, what="rows O")
        _close(l2[n], lse[b, h, i], atol=0, what="rows LSE")


def pin_diff(lib):
    """Differential attention: constant scores give (1 - lam) mean(V); lam = 0
    is vanilla with D_v = 128; identical streams give (1 - lam) vanilla."""
    S, H = 60, 2
    lam = 0.8
    qz = _bf(np.zeros((2, 1, S, H, 64)))
    k = _rand((2, 1, S, H, 64), "kd")
    v = _rand((1, S, H, 128), "vd")
    o, lse = oracle.diff_attention(qz, k, v, lam, lib=lib)
    _close(o, (1 - lam) * _f64(v).mean(axis=1, keepdims=True), what="diff closed form")
    _close(lse, math.log(S), what="diff LSE closed form")
    q = _rand((2, 1, S, H, 64), "qd")
    o, _ = oracle.diff_attention(q, k, v, 0.0, mask="causal", lib=lib)
    o0, _ = oracle.attention(q[0], k[0], v, mask="causal", lib=lib)
    _close(o, o0, atol=1e-12, what="diff lam 0")
    qq = np.ascontiguousarray(np.stack([q[0], q[0]]))
    kk = np.ascontiguousarray(np.stack([k[0], k[0]]))
    o, _ = oracle.diff_attention(qq, kk, v, lam, lib=lib)
    o0, _ = oracle.attention(q[0], k[0], v, lib=lib)
    _close(o, (1 - lam) * o0, atol=1e-12, what="diff identical streams")


def pin_evo(lib):
    """Evoformer: constant scores and zero bias give sigmoid(g) * mean(V);
    bias 0 with g = +50 is vanilla over the residue axis; the column pass is
    the row pass on the MSA tensor with its first two axes swapped."""
    Ns, Nr, H, c = 6, 40, 2, 32
    qz = _bf(np.zeros((Ns, Nr, H, c)))
    k, v, g = (_rand((Ns, Nr, H, c), n) for n in ("ke", "ve", "ge"))
    bias0 = _bf(np.zeros((H, Nr, Nr)))
    o, lse = oracle.evo_row(qz, k, v, bias0, g, lib=lib)
    sig = 1.0 / (1.0 + np.exp(-_f64(g)))
    _close(o, sig * _f64(v).mean(axis=1, keepdims=True), what="evo row closed form")
    _close(lse, math.log(Nr), what="evo LSE")
    q = _rand((Ns, Nr, H, c), "qe")
    g50 = _bf(np.full((Ns, Nr, H, c), 50.0))
    o, _ = oracle.evo_row(q, k, v, bias0, g50, lib=lib)
    o0, _ = oracle.attention(q, k, v, lib=lib)
    _close(o, o0, atol=1e-12, what="evo row = vanilla")
    oc, lc = oracle.evo_col(q, k, v, g, lib=lib)
    sw = lambda x: np.ascontiguousarray(np.swapaxes(x, 0, 1))
    bias_t = _bf(np.zeros((H, Ns, Ns)))
    orow, lrow = oracle.evo_row(sw(q), sw(k), sw(v), bias_t, sw(g), lib=lib)
    _close(oc, orow, atol=1e-12, what="evo col = row on transposed")
    _close(lc, lrow, atol=1e-12, what="evo col LSE")


def pin_composed_rows(lib):
    """The composed forms' sampled-row paths (Evoformer row and column passes,
    differential attention) equal the same rows of their full-tensor results,
    which the closed forms above pin.  N_seq = N_res = H here, so a gate gathered with
    its residue and head axes exchanged stays in bounds and gives other values;
    a second, larger shape has distinct extents on every axis.  The
    differential LSE of stream 0 is also compared with the plain attention of
    stream 0, which fixes the stream order."""
    for Ns, Nr, H in ((4, 4, 4), (7, 45, 3)):
        c = 32
        q, k, v, g = (_rand((Ns, Nr, H, c), n + f"cr{Nr}") for n in ("q", "k", "v", "g"))
        bias = _rand((H, Nr, Nr), f"bcr{Nr}")
        o, lse = oracle.evo_row(q, k, v, bias, g, lib=lib)
        rows = np.array([[s, h, i] for s in range(Ns) for h in range(H) for i in range(Nr)
                         if (s + 2 * h + 3 * i) % 4 == 0 or Nr == H])
        o2, l2 = oracle.evo_row(q, k, v, bias, g, rows=rows, lib=lib)
        for n, (s, h, i) in enumerate(rows):
            _close(o2[n], o[s, i, h], atol=0, what="evo row rows= O")
            _close(l2[n], lse[s, h, i], atol=0, what="evo row rows= LSE")
        oc, lc = oracle.evo_col(q, k, v, g, lib=lib)
        crow = np.array([[r, h, s] for r in range(Nr) for h in range(H) for s in range(Ns)
                         if (r + h + 2 * s) % 3 == 0 or Nr == H])
        oc2, lc2 = oracle.evo_col(q, k, v, g, rows=crow, lib=lib)
        for n, (r, h, s) in enumerate(crow):
            _close(oc2[n], oc[r, s, h], atol=0, what="evo col rows= O")
            _close(lc2[n], lc[r, h, s], atol=0, what="evo col rows= LSE")
    B, S, Hd = 2, 70, 3
    q = _rand((2, B, S, Hd, 64), "qcr")
    k = _rand((2, B, S, Hd, 64), "kcr")
    v = _rand((B, S, Hd, 128), "vcr")
    for mask in ("none", "causal"):
        o, lse = oracle.diff_attention(q, k, v, 0.8, mask=mask, lib=lib)
        _, l0 = oracle.attention(q[0], k[0], v, mask=mask, lib=lib)
        _close(lse[0], l0, atol=0, what="diff LSE stream 0")
        rows = np.array([[b, h, i] for b in range(B) for h in range(Hd) for i in range(0, S, 7)])
        o2, l2 = oracle.diff_attention(q, k, v, 0.8, mask=mask, rows=rows, lib=lib)
        for n, (b, h, i) in enumerate(rows):
            _close(o2[n], o[b, i, h], atol=0, what="diff rows= O")
            for st in range(2):
                _close(l2[st, n], lse[st, b, h, i], atol=0, what="diff rows= LSE")


def pin_fully_masked_row(lib):
    """A row with no allowed key (a document table whose first document starts
    after row 0 cannot occur in the workloads, so use prefix on Sq > Sk via a
    window of 0) returns O = 0 and LSE = -inf."""
    S = 10
    q, k, v = (_rand((1, S, 1, 64), n) for n in ("qm", "km", "vm"))
    o, lse = oracle.attention(q, k, v, mask="window", window=0, lib=lib)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse)), "fully masked rows"


def pin_decode(lib):
    """Serving with a KV cache: float64 SDPA with the boolean mask built from
    the definitions (query row i of a batch element with a cache of L keys sits
    at position L - Sq + i; KV-length: every key j < L), GQA, ragged lengths
    and Sq > 1; constant scores give the mean of V over keys 0..L-Sq+i and
    LSE ln(L-Sq+i+1); a cache of L keys equals attention over the first L keys
    alone; the decode mask with L = Sq = Sk is the causal mask; softcap."""
    B, Sq, Sk, Hq, Hk, D = 3, 4, 90, 8, 2, 64
    q = _rand((B, Sq, Hq, D), "qd")
    k, v = _rand((B, Sk, Hk, D), "kd"), _rand((B, Sk, Hk, D), "vd")
    L = np.array([90, 37, 4], dtype=np.int32)
    ii = np.arange(Sq)[None, :, None]
    jj = np.arange(Sk)[None, None, :]
    Lb = L[:, None, None]
    dec = (jj < Lb) & (jj <= Lb - Sq + ii)            # [B, Sq, Sk]
    kvl = np.broadcast_to(jj < Lb, (B, Sq, Sk))
    for name, m in (("decode", dec), ("kv_len", kvl)):
        o, _ = oracle.attention(q, k, v, mask=name, kv_len=L, lib=lib)
        ref = _sdpa(q, k, v, mask=torch.from_numpy(np.ascontiguousarray(m[:, None])),
                    enable_gqa=True)
        _close(o, ref, what=f"SDPA {name}")
    # closed form on constant scores
    q0 = _bf(np.zeros((B, Sq, Hq, D)))
    o, lse = oracle.attention(q0, k, v, mask="decode", kv_len=L, lib=lib)
    vf = _f64(v)
    for b in range(B):
        for i in range(Sq):
            n = int(L[b]) - Sq + i + 1
            for h in range(Hq):
                _close(o[b, i, h], vf[b, :n, h // (Hq // Hk)].mean(axis=0), what="decode mean")
                _close(lse[b, h, i], math.log(n), what="decode LSE")
    # a cache of L keys is attention over those L keys alone (per batch element)
    o, lse = oracle.attention(q, k, v, mask="kv_len", kv_len=L, lib=lib)
    for b in range(B):
        n = int(L[b])
        ob, lb = oracle.attention(q[b:b + 1], k[b:b + 1, :n], v[b:b + 1, :n], lib=lib)
        _close(o[b], ob[0], what="kv_len truncation")
        _close(lse[b], lb[0], what="kv_len truncation LSE")
    # decode with L = Sq = Sk is causal
    qs, ks, vs = _rand((2, 33, 2, D), "qs"), _rand((2, 33, 2, D), "ks"), _rand((2, 33, 2, D), "vs")
    o1, l1 = oracle.attention(qs, ks, vs, mask="decode", kv_len=np.array([33, 33]), lib=lib)
    o2, l2 = oracle.attention(qs, ks, vs, mask="causal", lib=lib)
    _close(o1, o2, what="decode = causal")
    _close(l1, l2, what="decode = causal LSE")
    # softcap on the decode mask against SDPA with the capped scores as an
    # additive term (scores computed in float64 from the same bits)
    cap = 20.0
    Q, K = _f64(q), _f64(k)
    z = np.einsum("bihd,bjhd->bhij", Q, np.repeat(K, Hq // Hk, axis=2)) / math.sqrt(D)
    add = cap * np.tanh(z / cap) - z + np.where(dec[:, None], 0.0, -np.inf)
    o, _ = oracle.attention(q, k, v, mod="softcap", softcap=cap, mask="decode", kv_len=L, lib=lib)
    _close(o, _sdpa(q, k, v, mask=torch.from_numpy(add), enable_gqa=True), atol=1e-9,
           what="SDPA decode softcap")


def pin_key_mask(lib):
    """The MSA key mask: removing a key by the mask equals deleting it from K,
    V and the bias (row and column passes), constant scores average V over the
    kept keys, an all-ones mask changes nothing, and a row with every key
    removed gives O = 0 and LSE = -inf."""
    Ns, Nr, H, c = 3, 90, 2, 32
    q, k, v = _rand((Ns, Nr, H, c), "mq"), _rand((Ns, Nr, H, c), "mk"), _rand((Ns, Nr, H, c), "mv")
    bias = _rand((H, Nr, Nr), "mb")
    rng = np.random.default_rng(5)
    mask = (rng.random((Ns, Nr)) > 0.3).astype(np.float32)
    mask[:, 0] = 1.0  # every MSA row keeps a residue
    mask[0, :] = 1.0  # every residue keeps an MSA row
    o, l = oracle.attention(q, k, v, bias=bias, key_mask=mask, lib=lib)
    for s in range(Ns):
        keep = np.nonzero(mask[s])[0]
        o2, l2 = oracle.attention(q[s:s + 1], np.ascontiguousarray(k[s:s + 1, keep]),
                                  np.ascontiguousarray(v[s:s + 1, keep]),
                                  bias=np.ascontiguousarray(bias[:, :, keep]), lib=lib)
        _close(o[s], o2[0], what=f"row pass, masked keys deleted (row {s})")
        _close(l[s], l2[0], what=f"row pass LSE (row {s})")
    # column pass: residue r attends over MSA rows t with mask[t, r] != 0
    g = _bf(np.zeros((Ns, Nr, H, c)))  # sigmoid(0) = 1/2 everywhere
    oc, lc = oracle.evo_col(q, k, v, g, msa_mask=mask, lib=lib)
    for r in (0, 7, 50, 89):
        keep = np.nonzero(mask[:, r])[0]
        o2, l2 = oracle.attention(np.ascontiguousarray(q[:, r:r + 1].swapaxes(0, 1)),
                                  np.ascontiguousarray(k[keep, r:r + 1].swapaxes(0, 1)),
                                  np.ascontiguousarray(v[keep, r:r + 1].swapaxes(0, 1)), lib=lib)
        _close(oc[r], 0.5 * o2[0], what=f"column pass, masked rows deleted (residue {r})")
        _close(lc[r], l2[0], what=f"column pass LSE (residue {r})")
    # constant scores: the mean of V over the kept keys
    z = _bf(np.zeros((Ns, Nr, H, c)))
    o, l = oracle.attention(z, k, v, key_mask=mask, lib=lib)
    vf = _f64(v)
    for s in range(Ns):
        keep = mask[s] != 0
        _close(o[s], np.broadcast_to(vf[s, keep].mean(axis=0), o[s].shape), what="constant scores")
        _close(l[s], math.log(keep.sum()), what="constant scores LSE")
    # all ones = no mask; a row with every key removed
    o1, l1 = oracle.attention(q, k, v, bias=bias, key_mask=np.ones((Ns, Nr)), lib=lib)
    o0, l0 = oracle.attention(q, k, v, bias=bias, lib=lib)
    _close(o1, o0, what="all-ones mask")
    mask[1] = 0.0
    o, l = oracle.attention(q, k, v, bias=bias, key_mask=mask, lib=lib)
    assert np.all(o[1] == 0.0) and np.all(np.isneginf(l[1])), "fully removed row"


def pin_backward(lib):
    """The backward oracle against float64 autograd of torch's
    scaled_dot_product_attention (MHA and GQA, with and without the causal
    mask, a non-default scale) and against central finite differences of the
    loss sum(dO * O) on a tiny problem."""
    for (B, S, Hq, Hk, D, mask, scale) in [(2, 37, 2, 2, 64, "none", 0.0), (1, 50, 4, 2, 64, "causal", 0.0),
                                           (1, 20, 2, 1, 16, "causal", 0.3)]:
        q, k, v = _rand((B, S, Hq, D), "bq"), _rand((B, S, Hk, D), "bk"), _rand((B, S, Hk, D), "bv")
        do = _rand((B, S, Hq, D), "bdo")
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, mask=mask, scale=scale)
        Q, K, V = (torch.from_numpy(_f64(x)).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, is_causal=mask == "causal", enable_gqa=Hq != Hk, scale=scale or None)
        o.backward(torch.from_numpy(_f64(do)).permute(0, 2, 1, 3))
        for name, mine, ref in (("dQ", dq, Q.grad), ("dK", dk, K.grad), ("dV", dv, V.grad)):
            _close(mine, ref.permute(0, 2, 1, 3).numpy(), atol=1e-10, what=f"backward {name} {mask}")
    # the other masks against autograd of SDPA with the same boolean mask
    B, S, Hq, Hk, D = 2, 70, 2, 1, 32
    q, k, v = _rand((B, S, Hq, D), "mq2"), _rand((B, S, Hk, D), "mk2"), _rand((B, S, Hk, D), "mv2")
    do = _rand((B, S, Hq, D), "mdo2")
    doc = np.array([[0, 13, 14, 50, S], [0, 40, S, S, S]], dtype=np.int32)
    for mask, kw in (("window", dict(window=9)), ("prefix", dict(prefix=21)), ("doc", dict(doc_offsets=doc))):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, mask=mask, **kw)
        allowed = np.stack([oracle._allowed(mask, S, b, kw.get("window", 0), kw.get("prefix", 0),
                                            kw.get("doc_offsets")) for b in range(B)])[:, None]
        Q, K, V = (torch.from_numpy(_f64(x)).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=torch.from_numpy(allowed),
                                                             enable_gqa=True)
        o.backward(torch.from_numpy(_f64(do)).permute(0, 2, 1, 3))
        for name, mine, ref in (("dQ", dq, Q.grad), ("dK", dk, K.grad), ("dV", dv, V.grad)):
            _close(mine, ref.permute(0, 2, 1, 3).numpy(), atol=1e-10, what=f"backward {name} {mask}")
        # the mask matrix itself from the interval form of each mask
        for b in range(B):
            for i in (0, 9, 21, 40, 69):
                lo, hi = _allowed_range(mask, i, S, kw.get("window", 0), kw.get("prefix", 0),
                                        list(doc[b][doc[b] < S]) if mask == "doc" else None)
                row = np.zeros(S, dtype=bool)
                row[lo:hi] = True
                assert np.array_equal(allowed[b, 0, i], row), f"{mask} row {i}"
    # ALiBi and softcap against autograd of the same forward written in torch
    B, S, Hq, Hk, D = 1, 50, 4, 2, 64
    q, k, v = _rand((B, S, Hq, D), "aq"), _rand((B, S, Hk, D), "ak"), _rand((B, S, Hk, D), "av")
    do = _rand((B, S, Hq, D), "ado")
    for mod in ("alibi", "softcap"):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, mod=mod, softcap=20.0, mask="causal")
        Q, K, V = (torch.from_numpy(_f64(x)).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
        Kr, Vr = K.repeat_interleave(Hq // Hk, dim=1), V.repeat_interleave(Hq // Hk, dim=1)
        u = (Q @ Kr.transpose(-1, -2)) / math.sqrt(D)
        if mod == "alibi":
            sl = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float64)
            dist = (torch.arange(S)[:, None] - torch.arange(S)[None, :]).abs().double()
            z = u - sl[None, :, None, None] * dist
        else:
            z = 20.0 * torch.tanh(u / 20.0)
        z = z.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
        o = torch.softmax(z, dim=-1) @ Vr
        o.backward(torch.from_numpy(_f64(do)).permute(0, 2, 1, 3))
        for name, mine, ref in (("dQ", dq, Q.grad), ("dK", dk, K.grad), ("dV", dv, V.grad)):
            _close(mine, ref.permute(0, 2, 1, 3).numpy(), atol=1e-10, what=f"backward {name} {mod}")
    # finite differences of L = sum(dO * O) with respect to one entry of each input
    B, S, Hq, Hk, D = 1, 6, 2, 1, 8
    q, k, v = _rand((B, S, Hq, D), "fq"), _rand((B, S, Hk, D), "fk"), _rand((B, S, Hk, D), "fv")
    do = _rand((B, S, Hq, D), "fdo")
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, mask="causal")
    Qf, Kf, Vf, dOf = _f64(q), _f64(k), _f64(v), _f64(do)

    def loss(Qx, Kx, Vx):
        tot = 0.0
        for h in range(Hq):
            z = (Qx[0, :, h] @ Kx[0, :, 0].T) / math.sqrt(D)
            z = np.where(np.tril(np.ones((S, S), dtype=bool)), z, -np.inf)
            p = np.exp(z - z.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            tot += float((dOf[0, :, h] * (p @ Vx[0, :, 0])).sum())
        return tot

    eps = 1e-6
    for name, grad, idx in (("dQ", dq, (0, 3, 1, 2)), ("dK", dk, (0, 2, 0, 5)), ("dV", dv, (0, 1, 0, 7))):
        args = [Qf.copy(), Kf.copy(), Vf.copy()]
        which = {"dQ": 0, "dK": 1, "dV": 2}[name]
        args[which][idx] += eps
        up = loss(*args)
        args[which][idx] -= 2 * eps
        down = loss(*args)
        _close(grad[idx], (up - down) / (2 * eps), atol=1e-7, what=f"finite difference {name}")


def pin_diff_backward(lib):
    """The differential backward against float64 autograd of the forward
    written in torch (both softmaxes, one V; MHA and GQA, with and without the
    causal mask, Dv 64 and 128, a non-default scale), and against two
    reductions: lambda = 0 is the plain backward of stream one (stream two's
    gradients vanish), and identical streams give (1 - lambda) times the plain
    backward for dV and the two streams' dQ, dK in the ratio 1 : -lambda."""
    for (B, S, H, Hk, D, Dv, mask, scale, lam) in [(2, 23, 2, 2, 16, 32, "none", 0.0, 0.8),
                                                   (1, 31, 4, 2, 16, 16, "causal", 0.3, 0.5)]:
        q, k = _rand((2, B, S, H, D), "dbq"), _rand((2, B, S, Hk, D), "dbk")
        v, do = _rand((B, S, Hk, Dv), "dbv"), _rand((B, S, H, Dv), "dbdo")
        dq, dk, dv = oracle.diff_attention_bwd(q, k, v, do, lam, mask=mask, scale=scale)
        Q, K = (torch.from_numpy(_f64(x)).permute(0, 1, 3, 2, 4).requires_grad_(True) for x in (q, k))
        V = torch.from_numpy(_f64(v)).permute(0, 2, 1, 3).requires_grad_(True)
        sc = scale or 1.0 / math.sqrt(D)
        Vr = V.repeat_interleave(H // Hk, dim=1)
        out = 0
        for t, c in ((0, 1.0), (1, -lam)):
            z = sc * (Q[t] @ K[t].repeat_interleave(H // Hk, dim=1).transpose(-1, -2))
            if mask == "causal":
                z = z.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
            out = out + c * (torch.softmax(z, dim=-1) @ Vr)
        out.backward(torch.from_numpy(_f64(do)).permute(0, 2, 1, 3))
        _close(dq, Q.grad.permute(0, 1, 3, 2, 4).numpy(), atol=1e-10, what=f"diff backward dQ {mask}")
        _close(dk, K.grad.permute(0, 1, 3, 2, 4).numpy(), atol=1e-10, what=f"diff backward dK {mask}")
        _close(dv, V.grad.permute(0, 2, 1, 3).numpy(), atol=1e-10, what=f"diff backward dV {mask}")
    # reductions, against the plain backward oracle
    B, S, H, Hk, D = 1, 40, 2, 1, 16
    q, k = _rand((2, B, S, H, D), "drq"), _rand((2, B, S, Hk, D), "drk")
    v, do = _rand((B, S, Hk, D), "drv"), _rand((B, S, H, D), "drdo")
    dq, dk, dv = oracle.diff_attention_bwd(q, k, v, do, 0.0, mask="causal")
    pq, pk, pv = oracle.attention_bwd(q[0], k[0], v, do, mask="causal")
    _close(dq[0], pq, atol=1e-12, what="diff backward lambda 0 dQ")
    _close(dk[0], pk, atol=1e-12, what="diff backward lambda 0 dK")
    _close(dv, pv, atol=1e-12, what="diff backward lambda 0 dV")
    _close(dq[1], 0 * pq, atol=1e-12, what="diff backward lambda 0 stream two")
    same_q, same_k = np.stack([q[0], q[0]]), np.stack([k[0], k[0]])
    lam = 0.3
    dq, dk, dv = oracle.diff_attention_bwd(same_q, same_k, v, do, lam, mask="causal")
    _close(dv, (1 - lam) * pv, atol=1e-12, what="diff backward identical streams dV")
    _close(dq[0], pq, atol=1e-12, what="diff backward identical streams dQ1")
    _close(dq[1], -lam * pq, atol=1e-12, what="diff backward identical streams dQ2")
    _close(dk[1], -lam * pk, atol=1e-12, what="diff backward identical streams dK2")


def pin_backward_expr(lib):
    """The backward with a score_mod expression: expressions that restate the
    built-in variants give the built-in backward, and the forward-mode
    derivative matches central differences of the expression's value."""
    from oracle import score_expr as se

    B, S, Hq, Hk, D = 1, 40, 4, 2, 32
    q, k, v = _rand((B, S, Hq, D), "eq"), _rand((B, S, Hk, D), "ek"), _rand((B, S, Hk, D), "ev")
    do = _rand((B, S, Hq, D), "edo")
    cases = [("score", "none", dict(mod="none")), ("20 * tanh(score / 20)", "none", dict(mod="softcap")),
             ("score - exp2(-8 * (h + 1) / 4) * abs(q_idx - kv_idx)", "causal", dict(mod="alibi")),
             ("where(kv_idx <= q_idx, score, -inf)", "none", dict(mod="none", mask="causal"))]
    for expr, mask, kw in cases:
        got = oracle.attention_bwd(q, k, v, do, mod="expr", expr=expr, mask=mask)
        kw = dict(kw)
        ref = oracle.attention_bwd(q, k, v, do, mask=kw.pop("mask", mask), **kw)
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            _close(a, b, atol=1e-10, what=f"expr backward {name} {expr!r}")
    rng = np.random.default_rng(9)
    x = rng.normal(size=200) * 3
    for expr in ["max(score, -2) * exp2(-h) + sqrt(abs(score) + 1) + log(2 + score * score) / (1 + score * score)",
                 "where(score > 0, tanh(score), exp(score) - 1) * (1 + 0.1 * floor(kv_idx / 3))",
                 "min(score, 1.5) - abs(score - 0.3) + log2(1 + exp(score))",
                 "exp2(score / 4) * sqrt(2 + score * score)"]:
        env = dict(b=1.0, h=2.0, q_idx=7.0, kv_idx=np.arange(200.0))
        _, d = se.evaluate_with_grad(expr, score=x, **env)
        eps = 1e-6
        fd = (se.evaluate(expr, score=x + eps, **env) - se.evaluate(expr, score=x - eps, **env)) / (2 * eps)
        kink = np.abs(x[:, None] - np.array([-2.0, 0.0, 0.3, 1.5])[None, :]).min(axis=1) < 1e-4
        _close(d[~kink], fd[~kink], atol=1e-5, what=f"derivative of {expr!r}")


def pin_score_expr(lib):
    """The score_mod-expression oracle (numpy, float64) against the C oracle's
    built-in variants written as expressions, against a closed form, on rows
    the expression removes entirely, and on the strings the grammar refuses."""
    from oracle import score_expr as se

    B, S, Hq, Hk, D = 2, 70, 4, 2, 64
    q, k, v = _rand((B, S, Hq, D), "xq"), _rand((B, S, Hk, D), "xk"), _rand((B, S, Hk, D), "xv")
    cases = [
        ("score", "none", dict(mod="none", mask="none")),
        ("score", "causal", dict(mod="none", mask="causal")),
        ("20 * tanh(score / 20)", "none", dict(mod="softcap", softcap=20.0, mask="none")),
        # default ALiBi slopes 2^(-8 (h + 1) / Hq) with Hq = 4
        ("score - exp2(-8 * (h + 1) / 4) * abs(q_idx - kv_idx)", "causal",
         dict(mod="alibi", mask="causal")),
        ("where(kv_idx <= q_idx, score, -inf)", "none", dict(mod="none", mask="causal")),
        ("where(kv_idx > q_idx, -inf, score)", "none", dict(mod="none", mask="causal")),
    ]
    for expr, mask, kw in cases:
        o, l = se.attention_expr(q, k, v, expr, mask=mask)
        o2, l2 = oracle.attention(q, k, v, lib=lib, **kw)
        _close(o, o2, atol=1e-9, what=f"expr {expr!r} O")
        _close(l, l2, atol=1e-9, what=f"expr {expr!r} LSE")
    # a constant logit c: O_i = mean of v over the allowed keys, LSE_i = c + ln(count)
    vf = _f64(v)
    csum = np.cumsum(vf, axis=1)
    o, l = se.attention_expr(q, k, v, "0 * score + 3", mask="causal")
    for h in range(Hq):
        cnt = np.arange(1, S + 1)[None, :, None]
        _close(o[:, :, h], csum[:, :, h // (Hq // Hk)] / cnt, what="constant logit O")
        _close(l[:, h], 3.0 + np.log(np.arange(1, S + 1))[None, :], what="constant logit LSE")
    # rows the expression removes entirely: O = 0, LSE = -inf; the others unchanged
    o, l = se.attention_expr(q, k, v, "where(q_idx < 5, -inf, score)")
    o2, l2 = se.attention_expr(q, k, v, "score")
    assert np.all(o[:, :5] == 0) and np.all(np.isneginf(l[:, :, :5]))
    _close(o[:, 5:], o2[:, 5:], what="unmasked rows")
    for bad in ["score ** 2", "score // 2", "a + 1", "1 < score < 3", "tanh(score, 1)", "tanh",
                "__import__('os')", "score if b else h", "[score]", "score.real", "True + score"]:
        try:
            se.parse(bad)
        except ValueError:
            continue
        raise AssertionError(f"the grammar accepted {bad!r}")


ALL_PINS = [pin_constant_scores, pin_alibi_geometric, pin_softcap_two_keys, pin_one_hot,
            pin_rows_sum_to_one, pin_shift_invariance, pin_permutation, pin_causal_row0,
            pin_sdpa, pin_reductions, pin_rows_api, pin_composed_rows, pin_diff, pin_evo, pin_fully_masked_row,
            pin_decode, pin_key_mask, pin_score_expr, pin_backward, pin_backward_expr,
            pin_diff_backward]
