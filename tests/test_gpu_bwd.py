"""GPU parity of the backward (dQ, dK, dV) with the float64 backward oracle.

The forward runs through the library (its bf16 O and fp32 LSE feed the
backward, as in training); the oracle differentiates the plain definition in
float64 from the same bf16 inputs.  Tolerance, derived from the arithmetic:
the MMA operands P and dS are rounded to bf16 (relative 2^-9 each), O enters
D = rowsum(dO O) rounded to bf16, and the gradients are rounded to bf16 on
output; summed over up to S terms of both signs these give errors of a few
2^-9 of the gradient's own scale.  D's rounding adds a term that does not
scale with the gradient: |delta_i| <= 2^-9 sum_d |dO_id O_id| enters dQ_i as
-scale delta_i sum_j P_ij k_j (and dK likewise), which matters where dS is
itself small, as in rows of two keys (dS_i0 = P_i0 P_i1 (dP_i0 - dP_i1)): a
two-key ALiBi row measured a mean error of 3.1 * 2^-9 of mean |dQ|.  So each
gradient must satisfy max |err| <= 10 * 2^-9 max |ref| and mean |err| <=
4 * 2^-9 mean |ref| (the mean bound is the tighter one where cancellation
leaves exact zeros, as in the first row of a causal dQ).
"""
import numpy as np
import pytest

import oracle
import testdata

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402

import attention_variant_gb300 as fa  # noqa: E402


def _run(tag, B, S, Hq, Hk, mask, mod="none", expr=None, **mkw):
    q = testdata.normal_bf16((B, S, Hq, 64), f"bwd_{tag}", "q")
    k = testdata.normal_bf16((B, S, Hk, 64), f"bwd_{tag}", "k")
    v = testdata.normal_bf16((B, S, Hk, 64), f"bwd_{tag}", "v")
    do = testdata.normal_bf16((B, S, Hq, 64), f"bwd_{tag}", "do")
    qd, kd, vd, dod = gu.dev(q), gu.dev(k), gu.dev(v), gu.dev(do)
    out = torch.empty((B, S, Hq, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    doc = mkw.pop("doc_offsets", None)
    doc_t = torch.from_numpy(doc).cuda() if doc is not None else None
    d = fa.make_desc(mask=mask, score_mod=mod, softcap=20.0, error_word=err, doc_offsets=doc_t, score_expr=expr,
                     **mkw)
    fa.fl_attn_fwd(qd, kd, vd, out, lse, d)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ws = torch.empty(fa.fl_attn_bwd_workspace_size(qd, kd, d), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the call must not depend on the workspace's contents
    fa.fl_attn_bwd(qd, kd, vd, out, lse, dod, dq, dk, dv, d, ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.attention_bwd(q, k, v, do, mod="expr" if expr else mod, expr=expr, softcap=20.0, mask=mask,
                               doc_offsets=doc, **mkw)
    return (gu.f64(dq), gu.f64(dk), gu.f64(dv)), ref


def _check(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        e = np.abs(g - r)
        assert e.max() <= 10 * 2.0 ** -9 * np.abs(r).max(), \
            f"{what} {name}: max err {e.max():.3e} vs max |ref| {np.abs(r).max():.3e}"
        assert e.mean() <= 4 * 2.0 ** -9 * np.abs(r).mean(), \
            f"{what} {name}: mean err {e.mean():.3e} vs mean |ref| {np.abs(r).mean():.3e}"


@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("B,S,Hq,Hk", [(2, 333, 2, 2), (1, 256, 8, 2), (1, 64, 2, 1), (1, 1000, 2, 2),
                                       (3, 5, 2, 2)])
def test_backward_matches_oracle(B, S, Hq, Hk, mask):
    got, ref = _run(f"{B}_{S}_{Hq}_{Hk}_{mask}", B, S, Hq, Hk, mask)
    _check(got, ref, f"B{B} S{S} Hq{Hq} Hk{Hk} {mask}")


@pytest.mark.parametrize("mask,kw", [("window", dict(window=100)), ("prefix", dict(prefix=150)),
                                     ("doc", None)])
@pytest.mark.parametrize("B,S,Hq,Hk", [(2, 333, 2, 2), (1, 700, 4, 2)])
def test_backward_other_masks(B, S, Hq, Hk, mask, kw):
    if mask == "doc":
        kw = dict(doc_offsets=testdata.doc_offsets(S, B, f"bwd_doc_{S}", 20, 200))
    got, ref = _run(f"{B}_{S}_{Hq}_{Hk}_{mask}", B, S, Hq, Hk, mask, **kw)
    _check(got, ref, f"B{B} S{S} Hq{Hq} Hk{Hk} {mask}")


@pytest.mark.parametrize("mod,mask,kw", [("alibi", "causal", {}), ("alibi", "none", {}),
                                         ("softcap", "none", {}), ("softcap", "window", dict(window=90))])
def test_backward_score_mods(mod, mask, kw):
    got, ref = _run(f"mod_{mod}_{mask}", 2, 333, 4, 2, mask, mod=mod, **kw)
    _check(got, ref, f"{mod} {mask}")


@pytest.mark.parametrize("expr,mask", [
    ("20 * tanh(score / 20)", "none"),
    ("score - 0.25 * abs(q_idx - kv_idx)", "causal"),
    ("where(kv_idx <= q_idx, score, -inf)", "none"),
    ("max(score, -1) + 0.5 * tanh(score) * (1 + 0.1 * h) + where(b == 1, 0.2, -0.1) * sqrt(abs(score) + 1)", "none"),
])
def test_backward_score_expressions(expr, mask):
    # the backward kernels compiled at run time with the expression and its
    # derivative (forward-mode, from the translator), against the oracle's
    # own forward-mode derivative
    got, ref = _run(f"expr_{testdata.fnv1a64(expr) % 997}", 2, 300, 4, 2, mask, expr=expr)
    _check(got, ref, f"expr {expr!r} {mask}")


def test_backward_is_deterministic():
    a, _ = _run("det", 1, 300, 4, 2, "causal")
    b, _ = _run("det", 1, 300, 4, 2, "causal")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
