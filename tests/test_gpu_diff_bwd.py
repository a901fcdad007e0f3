"""GPU parity of the differential-attention backward (dQ1, dQ2, dK1, dK2, dV)
with the float64 oracle.

The forward runs through the library (its per-stream fp32 LSE feeds the
backward, as in training); the oracle differentiates the plain definition in
float64 from the same bf16 inputs.  Tolerance: that of the standard backward
(max |err| <= 10 * 2^-9 max |ref|, mean |err| <= 4 * 2^-9 mean |ref| per
gradient; the mean bound covers the rounding of D = rowsum(dO O) from the
bf16 O, derived in tests/test_gpu_bwd.py), since each stream's partial
gradients come from the standard backward kernels; they are summed with their
coefficients in fp32 and rounded once, which adds at most one more bf16
rounding of a partial (2^-9 of its scale) where two partials meet (dV, and
dQ / dK at Dv = 128).
"""
import numpy as np
import pytest

import oracle
import testdata

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402

import attention_variant_gb300 as fa  # noqa: E402


def _run(tag, B, S, H, Hk, Dv, mask, lam):
    q = testdata.normal_bf16((2, B, S, H, 64), f"dbwd_{tag}", "q")
    k = testdata.normal_bf16((2, B, S, Hk, 64), f"dbwd_{tag}", "k")
    v = testdata.normal_bf16((B, S, Hk, Dv), f"dbwd_{tag}", "v")
    do = testdata.normal_bf16((B, S, H, Dv), f"dbwd_{tag}", "do")
    qd, kd, vd, dod = gu.dev(q), gu.dev(k), gu.dev(v), gu.dev(do)
    out = torch.empty((B, S, H, Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, B, H, S), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="diff", mask=mask, diff_lambda=lam, error_word=err)
    fa.fl_attn_fwd(qd, kd, vd, out, lse, d)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ws = torch.empty(fa.fl_attn_diff_bwd_workspace_size(qd, kd, vd, d), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the call must not depend on the workspace's contents
    fa.fl_attn_diff_bwd(qd, kd, vd, lse, dod, dq, dk, dv, d, ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.diff_attention_bwd(q, k, v, do, lam, mask=mask)
    return (gu.f64(dq), gu.f64(dk), gu.f64(dv)), ref


def _check(got, ref, what):
    names = ("dQ1", "dQ2", "dK1", "dK2", "dV")
    gq, gk, gv = got
    rq, rk, rv = ref
    for name, g, r in zip(names, (gq[0], gq[1], gk[0], gk[1], gv), (rq[0], rq[1], rk[0], rk[1], rv)):
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        e = np.abs(g - r)
        assert e.max() <= 10 * 2.0 ** -9 * np.abs(r).max(), \
            f"{what} {name}: max err {e.max():.3e} vs max |ref| {np.abs(r).max():.3e}"
        assert e.mean() <= 4 * 2.0 ** -9 * np.abs(r).mean(), \
            f"{what} {name}: mean err {e.mean():.3e} vs mean |ref| {np.abs(r).mean():.3e}"


@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("Dv", [64, 128])
@pytest.mark.parametrize("B,S,H,Hk", [(2, 333, 3, 3), (1, 256, 4, 2), (1, 130, 2, 1)])
def test_diff_backward_matches_oracle(B, S, H, Hk, Dv, mask):
    got, ref = _run(f"{B}_{S}_{H}_{Hk}_{Dv}_{mask}", B, S, H, Hk, Dv, mask, 0.8)
    _check(got, ref, f"diff backward B{B} S{S} H{H}/{Hk} Dv{Dv} {mask}")


@pytest.mark.parametrize("lam", [0.0, -1.5])
def test_diff_backward_lambda(lam):
    # lambda = 0: stream two's gradients are exactly zero; a negative lambda
    # adds the streams
    got, ref = _run(f"lam{lam}", 1, 200, 2, 2, 128, "causal", lam)
    _check(got, ref, f"diff backward lambda {lam}")
    if lam == 0.0:
        assert np.all(got[0][1] == 0) and np.all(got[1][1] == 0)


def test_diff_backward_several_items_per_cta():
    # 4 x 16 heads x 6 query blocks: every CTA of the inner kernels' persistent
    # grids runs several work items
    got, ref = _run("persist", 4, 700, 16, 16, 128, "causal", 0.8)
    _check(got, ref, "diff backward persistent")


def test_diff_backward_is_deterministic():
    a, _ = _run("det", 1, 300, 4, 2, 128, "none", 0.8)
    b, _ = _run("det", 1, 300, 4, 2, 128, "none", 0.8)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
