"""GPU parity of the differential-attention kernel against the CPU oracle.

O = softmax(scale Q1 K1^T) V - lambda softmax(scale Q2 K2^T) V with both
streams in one kernel; O max |err| <= 1e-2, mean <= 1e-3, per-stream LSE max
|err| <= 1e-3, visited-tile counts exact.
"""
import numpy as np
import pytest
import torch

import attention_variant_gb300 as fa
import oracle
import testdata
from testdata import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_variant_gb300 import build
    build.build()


def _inputs(tag, B, S, H, Hk=None, D=64, Dv=128):
    Hk = Hk or H
    q = testdata.normal_bf16((2, B, S, H, D), tag, "q")
    k = testdata.normal_bf16((2, B, S, Hk, D), tag, "k")
    v = testdata.normal_bf16((B, S, Hk, Dv), tag, "v")
    return q, k, v


def _bn(Dv):
    """Keys per key tile of the differential kernel for value head dimension Dv."""
    return fa.fl_attn_tile_shape(fa.make_desc(kind="diff"), Dv)[1]


def run_diff(q, k, v, lam, mask="none"):
    _, B, S, H, D = q.shape
    Dv = v.shape[3]
    out = torch.full((B, S, H, Dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.full((B, H, (S + 127) // 128), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="diff", mask=mask, diff_lambda=lam, debug_tile_counts=cnt,
                     error_word=err)
    fa.fl_attn_fwd(gu.dev(q), gu.dev(k), gu.dev(v), out, lse, d)
    torch.cuda.synchronize()
    return gu.f64(out), gu.f64(lse), cnt.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("S", [256, 333])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_diff_small(S, mask):
    q, k, v = _inputs(f"diff{S}", 2, S, 3)
    o, lse, cnt, err = run_diff(q, k, v, 0.8, mask)
    assert err == 0
    oref, lref = oracle.diff_attention(q, k, v, 0.8, mask=mask)
    gu.compare(o, lse, oref, lref, what=f"diff {S} {mask}")
    exp = gu.expected_tile_counts(mask, 2, 3, S, bn=_bn(128))
    assert np.array_equal(cnt, exp)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_diff_dv64(mask):
    # value head dimension 64 (one 64-column V half per key tile); 333 rows
    # leave a ragged last tile
    q, k, v = _inputs("diffdv64", 2, 333, 3, Dv=64)
    o, lse, cnt, err = run_diff(q, k, v, 0.8, mask)
    assert err == 0
    oref, lref = oracle.diff_attention(q, k, v, 0.8, mask=mask)
    gu.compare(o, lse, oref, lref, what=f"diff dv64 {mask}")
    assert np.array_equal(cnt, gu.expected_tile_counts(mask, 2, 3, 333, bn=_bn(64)))


def test_diff_dv64_full_size():
    """The differential workload's shape (B 4, S 4096, H 16) with Dv = 64,
    causal, rows at both ends of every query block against the oracle."""
    w = workloads.DIFF
    q, k, v = _inputs(w["name"] + "_dv64", w["B"], w["S"], w["H"], Dv=64)
    o, lse, cnt, err = run_diff(q, k, v, w["lam"], "causal")
    assert err == 0
    rows = gu.block_edge_rows(w["B"], w["H"], w["S"], n_random=64, seed=3)
    oref, lref = oracle.diff_attention(q, k, v, w["lam"], mask="causal", rows=rows)
    o_s = np.stack([o[b, i, h] for b, h, i in rows])
    l_s = np.stack([[lse[s, b, h, i] for b, h, i in rows] for s in range(2)])
    gu.compare(o_s, l_s, oref, lref, what="diff dv64 full causal")
    assert np.array_equal(cnt, gu.expected_tile_counts("causal", w["B"], w["H"], w["S"], bn=_bn(64)))


def test_diff_gqa_and_lambda_zero():
    q, k, v = _inputs("diffgqa", 1, 300, 4, 2)
    o, lse, _, _ = run_diff(q, k, v, 0.0, "causal")
    oref, lref = oracle.diff_attention(q, k, v, 0.0, mask="causal")
    gu.compare(o, lse, oref, lref, what="diff gqa lambda 0")


@pytest.mark.parametrize("Dv", [64, 128])
def test_diff_persistent_items_everywhere(Dv):
    # 320 work items: every CTA of the persistent grid runs two or more, so the
    # hand-over of both streams' O between items is exercised
    q, k, v = _inputs(f"diffpersist{Dv}", 4, 640, 16, Dv=Dv)
    for mask in ("none", "causal"):
        o, lse, cnt, err = run_diff(q, k, v, 0.8, mask)
        assert err == 0
        oref, lref = oracle.diff_attention(q, k, v, 0.8, mask=mask)
        gu.compare(o, lse, oref, lref, what=f"diff persistent dv{Dv} {mask}")
        assert np.array_equal(cnt, gu.expected_tile_counts(mask, 4, 16, 640, bn=_bn(Dv)))


@pytest.mark.parametrize("Dv", [64, 128])
@pytest.mark.parametrize("S", [1, 80, 112, 1000])
def test_diff_tile_edges(Dv, S):
    # lengths at and off both key-tile widths (80 and 112 keys), a single row
    q, k, v = _inputs(f"diffedge{S}", 1, S, 2, Dv=Dv)
    for mask in ("none", "causal"):
        o, lse, cnt, err = run_diff(q, k, v, 0.5, mask)
        assert err == 0
        oref, lref = oracle.diff_attention(q, k, v, 0.5, mask=mask)
        gu.compare(o, lse, oref, lref, what=f"diff edge S{S} dv{Dv} {mask}")
        assert np.array_equal(cnt, gu.expected_tile_counts(mask, 1, 2, S, bn=_bn(Dv)))


@pytest.mark.parametrize("Dv", [64, 128])
def test_diff_output_rows_off_32_byte_alignment(Dv):
    # O in a view 16 bytes into its buffer with a row pitch of Dv + 8
    # elements: the epilogue's 16-byte store path
    B, S, H = 1, 200, 2
    q, k, v = _inputs(f"diffmisal{Dv}", B, S, H, Dv=Dv)
    big = torch.full((B, S, H, Dv + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[..., 8:]
    lse = torch.full((2, B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fa.fl_attn_fwd(gu.dev(q), gu.dev(k), gu.dev(v), out, lse,
                   fa.make_desc(kind="diff", mask="causal", diff_lambda=0.5, error_word=err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oref, lref = oracle.diff_attention(q, k, v, 0.5, mask="causal")
    gu.compare(gu.f64(out), gu.f64(lse), oref, lref, what=f"diff misaligned rows dv{Dv}")
    assert torch.isnan(big[..., :8]).all()


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_diff_full_size(mask):
    """The whole output of the full-size workload against the oracle."""
    w = workloads.DIFF
    q, k, v = _inputs(w["name"], w["B"], w["S"], w["H"])
    o, lse, cnt, err = run_diff(q, k, v, w["lam"], mask)
    assert err == 0
    oref, lref = oracle.diff_attention(q, k, v, w["lam"], mask=mask)
    gu.compare(o, lse, oref, lref, what=f"diff full {mask}")
    assert np.array_equal(cnt, gu.expected_tile_counts(mask, w["B"], w["H"], w["S"], bn=_bn(128)))
