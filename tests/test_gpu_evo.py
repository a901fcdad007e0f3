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


def _bn(c):
    """Keys per key tile of the Evoformer kernel."""
    return fa.fl_attn_tile_shape(fa.make_desc(kind="evo_row"), c)[1]


def run_evo(row, q, k, v, g, bias, bias_pitch=None, lse_on=True):
    Ns, Nr, H, c = q.shape
    B, S = (Ns, Nr) if row else (Nr, Ns)
    out = torch.full((Ns, Nr, H, c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda") if lse_on else None
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
    return gu.f64(out), gu.f64(lse) if lse_on else None, cnt.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("Ns,Nr", [(4, 200), (3, 384), (5, 136)])
def test_evo_row_small(Ns, Nr):
    q, k, v, g, bias = _inputs(f"evo{Ns}_{Nr}", Ns, Nr, 2)
    o, lse, cnt, err = run_evo(True, q, k, v, g, bias)
    assert err == 0
    oref, lref = oracle.evo_row(q, k, v, bias, g)
    gu.compare(o, lse, oref, lref, what=f"evo row {Ns}x{Nr}")
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Ns, 2, Nr, bn=_bn(32)))


# c = 64 (the pages' Evoformer kernel benchmark: 4 heads of dimension 64;
# bias streamed per key tile) and c = 32 with N_res > 384 (bias streamed)
@pytest.mark.parametrize("Ns,Nr,c", [(4, 200, 64), (3, 384, 64), (3, 520, 32), (2, 712, 32),
                                     (2, 600, 64)])
def test_evo_row_streamed_bias(Ns, Nr, c):
    q, k, v, g, bias = _inputs(f"evos{Ns}_{Nr}_{c}", Ns, Nr, 2, c)
    o, lse, cnt, err = run_evo(True, q, k, v, g, bias)
    assert err == 0
    oref, lref = oracle.evo_row(q, k, v, bias, g)
    gu.compare(o, lse, oref, lref, what=f"evo row {Ns}x{Nr} c{c}")
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Ns, 2, Nr, bn=_bn(c)))


@pytest.mark.parametrize("Ns,Nr", [(200, 4), (130, 5)])
def test_evo_col_c64(Ns, Nr):
    q, k, v, g, _ = _inputs(f"evoc64_{Ns}_{Nr}", Ns, Nr, 2, 64)
    o, lse, cnt, err = run_evo(False, q, k, v, g, None)
    assert err == 0
    oref, lref = oracle.evo_col(q, k, v, g)
    gu.compare(o, lse, np.swapaxes(oref, 0, 1), lref, what=f"evo col c64 {Ns}x{Nr}")
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Nr, 2, Ns, bn=_bn(64)))


@pytest.mark.parametrize("c", [32, 64])
@pytest.mark.parametrize("row", [True, False], ids=["row", "col"])
def test_evo_persistent_items_everywhere(row, c):
    # several work items per CTA (odd chunks: one slot has a row fewer), and
    # the LSE-free path the benchmark times, compared everywhere
    Ns, Nr, H = (37, 256, 4) if row else (256, 37, 4)
    q, k, v, g, bias = _inputs(f"evop{int(row)}_{c}", Ns, Nr, H, c)
    for lse_on in (True, False):
        o, lse, cnt, err = run_evo(row, q, k, v, g, bias if row else None, lse_on=lse_on)
        assert err == 0
        if row:
            oref, lref = oracle.evo_row(q, k, v, bias, g)
        else:
            oref, lref = oracle.evo_col(q, k, v, g)
            oref = np.swapaxes(oref, 0, 1)
        gu.compare(o, lse, oref, lref if lse_on else None,
                   what=f"evo persistent {'row' if row else 'col'} c{c} lse={lse_on}")


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
    assert np.array_equal(cnt, gu.expected_tile_counts("none", Nr, 2, Ns, bn=_bn(32)))


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
    assert np.array_equal(cnt, gu.expected_tile_counts("none", B, H, S, bn=_bn(c)))


@pytest.mark.parametrize("row", [True, False], ids=["row", "col"])
def test_evo_c64_kernel_benchmark_shape(row):
    """The Evoformer kernel benchmark's head shape (4 heads of dimension 64)
    at the MSA size of the c = 32 workload (N_seq 512, N_res 384), the whole
    output against the oracle."""
    w = workloads.EVO_C64
    Ns, Nr, H, c = w["N_seq"], w["N_res"], w["H"], w["c"]
    q, k, v, g, bias = _inputs(w["name"], Ns, Nr, H, c)
    o, lse, cnt, err = run_evo(row, q, k, v, g, bias)
    assert err == 0
    if row:
        oref, lref = oracle.evo_row(q, k, v, bias, g)
    else:
        oref, lref = oracle.evo_col(q, k, v, g)
        oref = np.swapaxes(oref, 0, 1)
    gu.compare(o, lse, oref, lref, what="evo c64 " + ("row" if row else "col"))


@pytest.mark.parametrize("Ns,Nr,H,c", [(512, 520, 1, 32), (512, 384, 2, 64)])
def test_evo_streamed_bias_many_rows_per_slot(Ns, Nr, H, c):
    """Streamed bias with several MSA rows per slot in each work item, so the
    two slots' softmax warps release and the producer refills the bias stages
    at full pace.  (A stage released before the shared loads that read it had
    completed was refilled under the last warp to arrive: wrong logits in a few
    hundred rows, different from run to run.)  Two runs against one oracle
    result."""
    q, k, v, g, bias = _inputs(f"evosm{Nr}_{c}", Ns, Nr, H, c)
    oref, lref = oracle.evo_row(q, k, v, bias, g)
    for run in range(2):
        o, lse, cnt, err = run_evo(True, q, k, v, g, bias)
        assert err == 0
        gu.compare(o, lse, oref, lref, what=f"evo row streamed bias {Ns}x{Nr} c{c} run {run}")
