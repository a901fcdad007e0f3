"""fl_attn_decode_static: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc -- a serving loop that must not take the
device-wide synchronisation an allocation or a free can cause, or a plug-in
that does not own the process's device allocator -- and have no buffer to hand
over as a workspace.  fl_attn_decode_static serves them with the library's own
static scratch array (64 MiB).  Here it is called through the C ABI and
checked against fl_attn_decode (the same computation with a caller workspace)
on two calls in a row, since every call reuses the array the previous one
left behind; and a request larger than the array is refused with a clear
error.  This file is collected last, so a run that stops at its first failure
has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import attention_variant_gb300 as fa
import testdata

torch = pytest.importorskip("torch")

O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3  # the parity tolerances of every GPU test


def _paged_problem(B=4, Sq=2, Hq=8, Hk=2, lens=(1100, 257, 129, 5), page=64):
    per = [-(-L // page) for L in lens]
    n_pages = sum(per) + 2
    perm = np.random.default_rng(11).permutation(n_pages).astype(np.int32)
    table = np.full((B, max(per)), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        table[b, : per[b]] = perm[at: at + per[b]]
        at += per[b]
    to = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    q = to(testdata.normal_bf16((B, Sq, Hq, 64), "no_alloc", "q"))
    kp = to(testdata.normal_bf16((n_pages, page, Hk, 64), "no_alloc", "k"))
    vp = to(testdata.normal_bf16((n_pages, page, Hk, 64), "no_alloc", "v"))
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, kp, vp, lens_t, torch.from_numpy(table).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("mod", ["none", "softcap"])
def test_static_scratch_matches_workspace_call_twice(mod):
    q, kp, vp, lens_t, table_t = _paged_problem()
    B, Sq, Hq, _ = q.shape
    d = fa.make_decode_desc(lens_t, int(lens_t.max()), score_mod=mod, softcap=20.0, causal=True,
                            block_table=table_t)
    out_ref = torch.empty((B, Sq, Hq, 64), dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty((B, Hq, Sq), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fl_attn_decode_workspace_size(q, kp, d), dtype=torch.uint8, device="cuda")
    fa.fl_attn_decode(q, kp, vp, out_ref, lse_ref, d, ws)
    torch.cuda.synchronize()
    o_ref, l_ref = out_ref.float().cpu().numpy(), lse_ref.cpu().numpy()
    for call in range(2):
        out = torch.full((B, Sq, Hq, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        fa.fl_attn_decode_static(q, kp, vp, out, lse, d)
        torch.cuda.synchronize()
        o, l = out.float().cpu().numpy(), lse.cpu().numpy()
        err = np.abs(o.astype(np.float64) - o_ref)
        assert np.all(np.isfinite(o)), f"call {call}: non-finite output"
        assert err.max() <= O_MAX and err.mean() <= O_MEAN, f"call {call}: O differs by {err.max():.3e}"
        assert np.abs(l - l_ref).max() <= LSE_MAX, f"call {call}: LSE differs"


def test_static_scratch_refuses_oversize_requests():
    # 64 sequences x 64 KV heads x 32 chunks of 128 keys x 64 rows needs far more
    # than the 64 MiB array; refused before any device work
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
