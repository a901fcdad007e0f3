"""GPU parity of fl_attn_evoformer: batches of MSA stacks and the MSA mask.

Each stack is compared with the oracle's row or column pass on that stack
alone (the stacks are independent by definition), with the MSA mask removing
keys: residues of an MSA row in the row pass, MSA rows of a residue in the
column pass.  Masks are seeded, with ragged runs of removed keys, one fully
removed row (O = 0, LSE = -inf), and an all-kept stack.
"""
import numpy as np
import pytest
import torch

import attention_variant_gb300 as fa
import oracle
import testdata
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _stack_inputs(tag, Bt, Ns, Nr, H, c=32, per_stack_bias=True):
    q, k, v, g = (testdata.normal_bf16((Bt, Ns, Nr, H, c), tag, n) for n in ("q", "k", "v", "g"))
    bshape = (Bt, H, Nr, Nr) if per_stack_bias else (H, Nr, Nr)
    bias = testdata.normal_bf16(bshape, tag, "bias")
    return q, k, v, g, bias


def _mask(tag, Bt, Ns, Nr):
    """Seeded 0/1 mask [Bt, Ns, Nr]: ~25% removed, a removed run, stack 0 row 1
    removed entirely (row pass), stack Bt-1 all kept."""
    bits = testdata.normal_bf16((Bt, Ns, Nr), tag, "mask")
    m = (testdata.bf16_bits_to_f32(bits) > -0.67).astype(np.float32)
    m[:, :, 3:9] = 0.0
    m[:, 0, :] = 1.0  # every residue keeps MSA row 0 (column pass)
    m[:, :, 0] = 1.0  # every MSA row keeps residue 0 (row pass) ...
    m[0, 1, :] = 0.0  # ... except this one, removed entirely
    m[Bt - 1] = 1.0
    return m


def _run(row, q, k, v, g, bias, mask, mask_dtype=torch.float32):
    Bt, Ns, Nr, H, c = q.shape
    B, S = (Ns, Nr) if row else (Nr, Ns)
    out = torch.full((Bt, Ns, Nr, H, c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((Bt, B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = fa.make_desc(kind="evo_row" if row else "evo_col", error_word=err)
    m_t = torch.from_numpy(mask).to("cuda", mask_dtype) if mask is not None else None
    fa.fl_attn_evoformer(gu.dev(q), gu.dev(k), gu.dev(v), out, lse, d,
                         bias=gu.dev(bias) if row else None, gate=gu.dev(g), msa_mask=m_t)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return gu.f64(out), gu.f64(lse)


@pytest.mark.parametrize("per_stack_bias", [True, False])
@pytest.mark.parametrize("mask_dtype", [torch.float32, torch.bfloat16])
def test_row_pass_batched_masked(per_stack_bias, mask_dtype):
    Bt, Ns, Nr, H = 3, 4, 200, 2
    q, k, v, g, bias = _stack_inputs(f"rowb{int(per_stack_bias)}", Bt, Ns, Nr, H,
                                     per_stack_bias=per_stack_bias)
    mask = _mask("rowmask", Bt, Ns, Nr)
    o, lse = _run(True, q, k, v, g, bias, mask, mask_dtype)
    for b in range(Bt):
        bb = bias[b] if per_stack_bias else bias
        oref, lref = oracle.evo_row(q[b], k[b], v[b], bb, g[b], msa_mask=mask[b])
        gu.compare(o[b], lse[b], oref, lref, what=f"row pass stack {b}")
    assert np.all(o[0, 1] == 0.0) and np.all(np.isneginf(lse[0, 1]))


def test_column_pass_batched_masked():
    Bt, Ns, Nr, H = 2, 300, 5, 2
    q, k, v, g, _ = _stack_inputs("colb", Bt, Ns, Nr, H)
    mask = _mask("colmask", Bt, Ns, Nr)
    o, lse = _run(False, q, k, v, g, None, mask)
    for b in range(Bt):
        oref, lref = oracle.evo_col(q[b], k[b], v[b], g[b], msa_mask=mask[b])
        # the kernel writes O in the [N_seq, N_res, H, c] layout of its inputs
        gu.compare(np.swapaxes(o[b], 0, 1), lse[b], oref, lref, what=f"column pass stack {b}")


def test_unbatched_mask_through_the_same_entry_point():
    Ns, Nr, H = 3, 384, 2
    q, k, v, g, bias = _stack_inputs("row1", 1, Ns, Nr, H, per_stack_bias=False)
    mask = _mask("row1mask", 1, Ns, Nr)[0]
    out = torch.empty((Ns, Nr, H, 32), dtype=torch.bfloat16, device="cuda")
    d = fa.make_desc(kind="evo_row")
    fa.fl_attn_evoformer(gu.dev(q[0]), gu.dev(k[0]), gu.dev(v[0]), out, None, d,
                         bias=gu.dev(bias), gate=gu.dev(g[0]),
                         msa_mask=torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    oref, _ = oracle.evo_row(q[0], k[0], v[0], bias, g[0], msa_mask=mask)
    gu.compare(gu.f64(out), None, oref, None, what="unbatched masked row pass")


def test_batched_without_mask_matches_single_calls():
    Bt, Ns, Nr, H = 2, 3, 136, 2
    q, k, v, g, bias = _stack_inputs("nomask", Bt, Ns, Nr, H)
    o, lse = _run(True, q, k, v, g, bias, None)
    for b in range(Bt):
        oref, lref = oracle.evo_row(q[b], k[b], v[b], bias[b], g[b])
        gu.compare(o[b], lse[b], oref, lref, what=f"unmasked stack {b}")


def test_batched_shape_errors_launch_nothing():
    Bt, Ns, Nr, H = 2, 2, 64, 2
    q, k, v, g, bias = _stack_inputs("bad", Bt, Ns, Nr, H)
    out = torch.full((Bt, Ns, Nr, H, 32), 7.0, dtype=torch.bfloat16, device="cuda")
    d = fa.make_desc(kind="evo_row")
    bad_mask = torch.ones((Bt, Ns, Nr + 1), device="cuda")
    with pytest.raises(fa.FlAttnError):
        fa.fl_attn_evoformer(gu.dev(q), gu.dev(k), gu.dev(v), out, None, d, bias=gu.dev(bias),
                             gate=gu.dev(g), msa_mask=bad_mask)
    with pytest.raises(fa.FlAttnError):  # a stack count that differs
        fa.fl_attn_evoformer(gu.dev(q), gu.dev(k[:1]), gu.dev(v), out, None, d, bias=gu.dev(bias),
                             gate=gu.dev(g))
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call wrote the output"


@pytest.mark.parametrize("row", [True, False])
def test_batched_masked_c64(row):
    Bt, Ns, Nr, H = 2, 5, 200, 2
    if not row:
        Ns, Nr = 200, 5
    q, k, v, g, bias = _stack_inputs(f"c64b{int(row)}", Bt, Ns, Nr, H, c=64)
    mask = _mask(f"c64mask{int(row)}", Bt, Ns, Nr)
    o, lse = _run(row, q, k, v, g, bias, mask)
    for b in range(Bt):
        if row:
            oref, lref = oracle.evo_row(q[b], k[b], v[b], bias[b], g[b], msa_mask=mask[b])
            gu.compare(o[b], lse[b], oref, lref, what=f"c64 row stack {b}")
        else:
            oref, lref = oracle.evo_col(q[b], k[b], v[b], g[b], msa_mask=mask[b])
            gu.compare(np.swapaxes(o[b], 0, 1), lse[b], oref, lref, what=f"c64 col stack {b}")


@pytest.mark.parametrize("row", [True, False])
def test_af2_batched_workload_everywhere(row):
    # the benchmark's batch of masked AlphaFold2-sized stacks, at full size;
    # every stack's whole output against the oracle
    import bench

    e = bench.evo_batched_entry(row)
    Bt, Ns, Nr, H, c = e["Bt"], e["Ns"], e["Nr"], e["H"], e["c"]
    shape = (Bt, Ns, Nr, H, c)
    q, k, v, g = (testdata.normal_bf16(shape, e["name"], n) for n in "qkvg")
    bias = testdata.normal_bf16((Bt, H, Nr, Nr), e["name"], "bias") if row else None
    o, lse = _run(row, q, k, v, g, bias, e["mask"])
    for b in range(Bt):
        if row:
            oref, lref = oracle.evo_row(q[b], k[b], v[b], bias[b], g[b], msa_mask=e["mask"][b])
            og = o[b]
        else:
            oref, lref = oracle.evo_col(q[b], k[b], v[b], g[b], msa_mask=e["mask"][b])
            og = np.swapaxes(o[b], 0, 1)
        gu.compare(og, lse[b], oref, lref, what=f"af2 {'row' if row else 'col'} stack {b}")
