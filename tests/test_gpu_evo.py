"""GPU parity of the Evoformer row- and column-wise gated attention kernel
against the CPU oracle (O max |err| <= 1e-2, mean <= 1e-3, LSE max <= 1e-3,
visited-tile counts exact)."""
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


def _inputs(tag, Ns, Nr, H, c=32):
    q, k, v, g = (testdata.normal_bf16((Ns, Nr, H, c), tag, n) for n in ("q", "k", "v", "g"))
    bias = testdata.normal_bf16((H, Nr, Nr), tag, "bias")
    return q, k, v, g, bias


def run_evo(row, q, k, v, g, bias, bias_pitch=None):
    Ns, Nr, H, c = q.shape
    B, S = (Ns, Nr) if row else (Nr, Ns)
    out = torch.full((Ns, Nr, H, c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    cnt = torch.full((B, H, (S + 127) // 128), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="evo_row" if row else "evo_col", debug_tile_counts=cnt, error_word=err)
    bias_t = None
    if row:
        if bias_pitch is None:
            bias_t = gu.dev(bias)
        else:  # rows padded to bias_pitch elements (a strided, 16-byte aligned view)
            H = bias.shape[0]
            padded = np.zeros((H, Nr, bias_pitch), dtype=np.uint16)
            padded[:, :, :Nr] = bias
            bias_t = gu.dev(padded)[:, :, :Nr]
    fa.fl_attn_fwd(gu.dev(q), gu.dev(k), gu.dev(v), out, lse, d, bias=bias_t, gate=gu.dev(g))
    torch.cuda.synchronize()
    return gu.f64(out), gu.f64(lse), cnt.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("Ns,Nr", [(4, 200), (3, 384), (5, 136)])
def test_evo_row_small(Ns, Nr):
    q, k, v, g, bias = _inputs(f"evo{Ns}_{Nr}", Ns, Nr, 2)
    o, lse, cnt, err = run_evo(True, q, k, v, g, bias)
    assert err == 0
    oref, lref = oracle.evo_row(q, k, v, bias, g)
    gu.compare(o, lse, oref, lref, what=f"evo row {Ns}x{Nr}")
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Ns, 2, Nr))


def test_evo_row_ragged_padded_bias():
    """N_res = 130: the bias rows are padded to a 16-byte multiple (pitch 136)
    and passed as a strided view; the last key tile is ragged."""
    q, k, v, g, bias = _inputs("evopad", 3, 130, 2)
    o, lse, cnt, err = run_evo(True, q, k, v, g, bias, bias_pitch=136)
    assert err == 0
    oref, lref = oracle.evo_row(q, k, v, bias, g)
    gu.compare(o, lse, oref, lref, what="evo row padded bias")


def test_evo_rejects_unaligned_bias():
    q, k, v, g, bias = _inputs("evobad", 2, 130, 2)
    with pytest.raises(fa.FlAttnError) as e:
        run_evo(True, q, k, v, g, bias)
    assert e.value.status == fa.FL_ERR_ALIGNMENT


@pytest.mark.parametrize("Ns,Nr", [(200, 4), (512, 3), (130, 5)])
def test_evo_col_small(Ns, Nr):
    q, k, v, g, _ = _inputs(f"evoc{Ns}_{Nr}", Ns, Nr, 2)
    o, lse, cnt, err = run_evo(False, q, k, v, g, None)
    assert err == 0
    oref, lref = oracle.evo_col(q, k, v, g)
    gu.compare(o, lse, np.swapaxes(oref, 0, 1), lref, what=f"evo col {Ns}x{Nr}")
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Nr, 2, Ns))


@pytest.mark.parametrize("row", [True, False], ids=["row", "col"])
def test_evo_full_size(row):
    w = workloads.EVO
    Ns, Nr, H, c = w["N_seq"], w["N_res"], w["H"], w["c"]
    q, k, v, g, bias = _inputs(w["name"], Ns, Nr, H, c)
    o, lse, cnt, err = run_evo(row, q, k, v, g, bias)
    assert err == 0
    B, S = (Ns, Nr) if row else (Nr, Ns)
    # the whole output against the oracle
    if row:
        oref, lref = oracle.evo_row(q, k, v, bias, g)
    else:
        oref, lref = oracle.evo_col(q, k, v, g)
        oref = np.swapaxes(oref, 0, 1)
    gu.compare(o, lse, oref, lref, what="evo full " + ("row" if row else "col"))
    assert np.array_equal(cnt, gu.expected_tile_counts("none", B, H, S))
