"""The C-ABI library on the host: it loads, exports every declared symbol,
and rejects bad requests before touching any device (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import attention_variant_gb300 as fa
from attention_variant_gb300 import build as fbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fl_attn.h")


def _gpu_visible():
    try:
        import torch
    except ImportError:
        return False
    return torch.cuda.is_available()


# Tests that pass made-up device addresses: each call is refused before any
# device work, but on a machine with a GPU a call that validation accepted
# would launch on them, so these run only where no GPU is visible.
fake_addresses = pytest.mark.skipif(_gpu_visible(), reason="made-up device addresses (host-only test)")


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fl_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "fl_attn_fwd" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fl_attn.h but not exported"


def test_version_and_strings(lib):
    assert fa.fl_attn_version() == 1
    for s in range(7):
        assert fa.fl_attn_status_string(s).startswith("FL_")


def _t(shape, dtype=fa.FL_BF16, ptr=0x10000, strides=None):
    t = fa.FlTensor()
    t.ptr = ptr
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for d, (s, st) in enumerate(zip(shape, strides)):
        t.sizes[d] = s
        t.strides[d] = st
    return t


def _call(lib, q, k, v, o, lse=None, desc=None, bias=None, gate=None):
    desc = desc or fa.make_desc()
    r = lambda x: ctypes.byref(x) if x is not None else None
    return lib.fl_attn_fwd(r(q), r(k), r(v), r(o), r(lse), ctypes.byref(desc), r(bias), r(gate),
                           None)


@fake_addresses
def test_validation_before_device(lib):
    B, S, H, D = 2, 256, 4, 64
    good = lambda: _t((B, S, H, D))
    # every failure below happens before any CUDA call
    assert _call(lib, None, good(), good(), good()) == fa.FL_ERR_INVALID_ARG
    assert "q is NULL" in fa.fl_attn_last_error()
    assert _call(lib, good(), _t((B, S + 1, H, D)), good(), good()) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), _t((B, S, H, D), dtype=fa.FL_F32)) == \
        fa.FL_ERR_INVALID_ARG
    assert _call(lib, _t((B, S, H, D), ptr=0x10008), good(), good(), good()) == fa.FL_ERR_ALIGNMENT
    odd = _t((B, S, H, D), strides=(S * H * D, H * D + 4, D, 1))
    assert _call(lib, odd, good(), good(), good()) == fa.FL_ERR_ALIGNMENT
    notinner = _t((B, S, H, D), strides=(S * H * D, H * D, D, 2))
    assert _call(lib, notinner, good(), good(), good()) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, _t((B, S, H, 96)), _t((B, S, H, 96)), _t((B, S, H, 96)),
                 _t((B, S, H, 96))) == fa.FL_ERR_UNSUPPORTED  # head dimension
    assert _call(lib, _t((B, S, H, 64)), _t((B, S, H, 64)), _t((B, S, H, 128)),
                 _t((B, S, H, 128))) == fa.FL_ERR_UNSUPPORTED  # D != Dv
    # 2^31 work items or more (the kernel decodes item indices in 32 bits):
    # 2^20 batches x 16 heads x 256 pairs of query blocks
    huge = lambda: _t((1 << 20, 1 << 16, 16, D))
    assert _call(lib, huge(), huge(), huge(), huge()) == fa.FL_ERR_UNSUPPORTED
    assert "work items" in fa.fl_attn_last_error()
    assert _call(lib, _t((B, S, 3, D)), _t((B, S, 2, D)), _t((B, S, 2, D)),
                 _t((B, S, 3, D))) == fa.FL_ERR_INVALID_ARG  # Hq % Hk
    assert _call(lib, good(), good(), good(), good(),
                 desc=fa.make_desc(mask="window", window=0)) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(),
                 desc=fa.make_desc(mask="doc")) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(),
                 desc=fa.make_desc(score_mod="softcap", softcap=0.0)) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(),
                 desc=fa.make_desc(gqa_group=2)) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(), lse=_t((B, H, S + 1), fa.FL_F32)) == \
        fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(), bias=_t((H, S, S))) == fa.FL_ERR_INVALID_ARG
    assert _call(lib, good(), good(), good(), good(), desc=fa.make_desc(kind=7)) == \
        fa.FL_ERR_INVALID_ARG


def test_size_one_axes_take_any_stride(lib):
    # a size-1 axis may carry any stride (torch often reports 1 there).  With a
    # GPU the call runs, on real buffers of the extent the strides address;
    # without one it stops at the device lookup, after validation.
    n = 256 * 64
    if _gpu_visible():
        import torch
        bufs = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
        ptrs = [b.data_ptr() for b in bufs]
    else:
        ptrs = [0x10000 + 2 * n * i for i in range(4)]
    q, k, v, o = (_t((1, 256, 1, 64), ptr=p, strides=(1, 64, 1, 1)) for p in ptrs)
    st = _call(lib, q, k, v, o)
    if _gpu_visible():
        torch.cuda.synchronize()
        assert st == fa.FL_OK, fa.fl_attn_last_error()
    else:
        assert st not in (fa.FL_ERR_ALIGNMENT, fa.FL_ERR_INVALID_ARG), fa.fl_attn_last_error()


def test_tile_shape(lib):
    assert fa.fl_attn_tile_shape(fa.make_desc(), 64) == (128, 112)
    assert fa.fl_attn_tile_shape(fa.make_desc(), 32) == (128, 128)
    assert fa.fl_attn_tile_shape(fa.make_desc(), 128) == (128, 64)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="diff"), 64) == (128, 112)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="diff"), 128) == (128, 80)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="evo_row"), 32) == (128, 128)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="evo_col"), 64) == (128, 128)
    with pytest.raises(fa.FlAttnError):
        fa.fl_attn_tile_shape(fa.make_desc(), 48)


def _ddesc(max_kv=1000, kv_lens=0x20000, block_table=None, bt_stride=0, score_mod=0, softcap=0.0):
    d = fa.FlDecodeDesc()
    d.score_mod = score_mod
    d.softcap = softcap
    d.causal = 1
    d.kv_lens = kv_lens
    d.max_kv_len = max_kv
    d.block_table = block_table
    d.block_table_stride = bt_stride
    return d


def _ws_bytes(lib, q, kc, d):
    n = ctypes.c_size_t()
    st = lib.fl_attn_decode_workspace_size(ctypes.byref(q), ctypes.byref(kc), ctypes.byref(d),
                                           ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("B,Sq,Hq,Hk,Smax,split_keys", [
    (3, 2, 8, 2, 1000, 128),     # few sequences: the shortest splits
    (64, 1, 32, 8, 8192, 1024),  # 512 (sequence, KV head) pairs x 8 splits of 1024 >= 2048
    (16, 1, 32, 8, 8192, 512),   # 128 pairs x 8 splits of 1024 < 2048; x 16 of 512 = 2048
    (4, 1, 32, 8, 8192, 128),    # 32 pairs x 64 splits of 128 = 2048
])
def test_decode_workspace_size(lib, B, Sq, Hq, Hk, Smax, split_keys):
    # one fp32 partial (64 outputs, max, sum) per (sequence, KV head, split,
    # query row) and one counter per (sequence, KV head), each 256-byte aligned
    st, n = _ws_bytes(lib, _t((B, Sq, Hq, 64)), _t((B, Smax, Hk, 64)), _ddesc(max_kv=Smax))
    assert st == fa.FL_OK, fa.fl_attn_last_error()
    R, splits = (Hq // Hk) * Sq, -(-Smax // split_keys)
    up = lambda x: -(-x // 256) * 256
    units = B * Hk * splits * R
    assert n == up(units * 64 * 4) + up(units * 2 * 4) + up(B * Hk * 4)


@fake_addresses
def test_decode_validation_before_device(lib):
    B, Sq, Hq, Hk, Smax = 2, 1, 8, 2, 512
    q, kc = _t((B, Sq, Hq, 64)), _t((B, Smax, Hk, 64))
    r = lambda x: ctypes.byref(x) if x is not None else None

    def call(q=q, kc=kc, vc=None, o=None, lse=None, d=None, ws=0x40000, nbytes=1 << 30):
        vc = vc if vc is not None else _t((B, Smax, Hk, 64))
        o = o if o is not None else _t((B, Sq, Hq, 64))
        d = d if d is not None else _ddesc(max_kv=500)
        return lib.fl_attn_decode(r(q), r(kc), r(vc), r(o), r(lse), ctypes.byref(d), ws, nbytes,
                                  None)

    assert _ws_bytes(lib, _t((B, Sq, Hq, 128)), _t((B, Smax, Hk, 128)), _ddesc())[0] == \
        fa.FL_ERR_UNSUPPORTED                                        # head dimension
    assert _ws_bytes(lib, _t((B, 17, Hq, 64)), kc, _ddesc(max_kv=500))[0] == \
        fa.FL_ERR_UNSUPPORTED                                        # (Hq/Hk) * Sq > 64
    assert _ws_bytes(lib, q, kc, _ddesc(max_kv=513))[0] == fa.FL_ERR_INVALID_ARG  # > S_max
    assert _ws_bytes(lib, q, _t((5, 48, Hk, 64)), _ddesc(max_kv=500, block_table=0x30000,
                                                         bt_stride=11))[0] == fa.FL_ERR_UNSUPPORTED
    assert _ws_bytes(lib, q, _t((5, 64, Hk, 64)), _ddesc(max_kv=500, block_table=0x30000,
                                                         bt_stride=7))[0] == fa.FL_ERR_INVALID_ARG
    assert _ws_bytes(lib, q, kc, _ddesc(max_kv=500, score_mod=fa.FL_MOD_ALIBI))[0] == \
        fa.FL_ERR_UNSUPPORTED
    assert _ws_bytes(lib, q, kc, _ddesc(max_kv=500, score_mod=fa.FL_MOD_SOFTCAP))[0] == \
        fa.FL_ERR_INVALID_ARG                                        # softcap 0
    assert call(vc=_t((B, Smax, Hk + 1, 64))) == fa.FL_ERR_INVALID_ARG
    assert call(ws=0) == fa.FL_ERR_INVALID_ARG
    assert call(ws=0x40010) == fa.FL_ERR_ALIGNMENT
    assert call(nbytes=1024) == fa.FL_ERR_INVALID_ARG
    assert "workspace holds" in fa.fl_attn_last_error()
    assert call(o=_t((B, Sq, Hq + 1, 64))) == fa.FL_ERR_INVALID_ARG
    assert call(lse=_t((B, Hq, Sq + 1), fa.FL_F32)) == fa.FL_ERR_INVALID_ARG
    assert call(d=_ddesc(max_kv=500, kv_lens=None)) == fa.FL_ERR_INVALID_ARG


# ---- score_mod expressions (FL_MOD_EXPR)

GOOD_EXPRS = ["score", "20 * tanh(score / 20)", "score - 0.5 * abs(q_idx - kv_idx)",
              "where(kv_idx <= q_idx, score, -inf)", "max(score, .5e1) + (q_idx >= kv_idx) * 2",
              "exp2(-(h + 1) / 2) * floor(kv_idx / 64) + log(1 + exp(score)) - sqrt(b + 1) + log2(4)",
              "min(score, 3.) / 2 - +score * -1"]
BAD_EXPRS = ["", "score +", "score ** 2", "score // 2", "score /* c */", "a + 1", "1 < score < 3",
             "tanh(score, 1)", "tanh", "where(score, 1)", "20f", "1e", "0x10", "score; score",
             "score = 1", "(score", "score)", "score & 1", "score ? 1 : 0", "pi * score"]


@pytest.mark.parametrize("expr", GOOD_EXPRS)
def test_score_expr_grammar_accepts(lib, expr):
    assert lib.fl_attn_score_expr_check(expr.encode(), 0) == fa.FL_OK, fa.fl_attn_last_error()


@pytest.mark.parametrize("expr", BAD_EXPRS)
def test_score_expr_grammar_refuses(lib, expr):
    assert lib.fl_attn_score_expr_check(expr.encode(), 0) == fa.FL_ERR_INVALID_ARG
    assert "score_mod_expr" in fa.fl_attn_last_error()


def test_score_expr_grammar_matches_the_oracle_grammar():
    # the CUDA translator and the oracle's parser are separate code; every
    # string one accepts the other accepts, and the same for refusals
    from oracle import score_expr as se

    for expr in GOOD_EXPRS:
        se.parse(expr)
    for expr in BAD_EXPRS:
        if expr in ("0x10",):  # a Python literal the CUDA side refuses: stricter there
            continue
        with pytest.raises(ValueError):
            se.parse(expr)


def test_score_expr_runtime_compilation_needs_no_device(lib):
    # the whole standard kernel is compiled for sm_103a with the expression
    # as its score_mod (NVRTC; no GPU involved)
    st = lib.fl_attn_score_expr_check(b"score - 0.25 * abs(q_idx - kv_idx) + h * b", 1)
    assert st == fa.FL_OK, fa.fl_attn_last_error()


@fake_addresses
def test_score_expr_refused_before_device(lib):
    B, S, H, D = 2, 256, 4, 64
    t = lambda: _t((B, S, H, D))
    d = fa.make_desc(score_expr="score ** 2")
    assert _call(lib, t(), t(), t(), t(), desc=d) == fa.FL_ERR_INVALID_ARG
    assert "score_mod_expr" in fa.fl_attn_last_error()
    d = fa.make_desc(score_mod="expr")  # no string
    assert _call(lib, t(), t(), t(), t(), desc=d) == fa.FL_ERR_INVALID_ARG
    # the other kinds take no expression
    d = fa.make_desc(kind="evo_row", score_expr="score")
    assert _call(lib, _t((4, 64, 8, 32)), _t((4, 64, 8, 32)), _t((4, 64, 8, 32)),
                 _t((4, 64, 8, 32)), desc=d) != fa.FL_OK


def test_evoformer_batched_validation_before_device(lib):
    Bt, Ns, Nr, H, c = 2, 4, 64, 2, 32
    t5 = lambda: _t((Bt, Ns, Nr, H, c))
    r = lambda x: ctypes.byref(x) if x is not None else None

    def call(q=None, k=None, bias=None, mask=None, kind="evo_row"):
        d = fa.make_desc(kind=kind)
        q, k = q or t5(), k or t5()
        return lib.fl_attn_evoformer(r(q), r(k), r(t5()), r(t5()), None, ctypes.byref(d), r(bias),
                                     r(t5()), r(mask), None)

    assert call(kind="standard") == fa.FL_ERR_INVALID_ARG
    assert call(k=_t((Bt + 1, Ns, Nr, H, c))) == fa.FL_ERR_INVALID_ARG
    assert "stacks" in fa.fl_attn_last_error()
    assert call(bias=_t((Bt, H, Nr, Nr)), mask=_t((Bt, Ns, Nr + 1), dtype=fa.FL_F32)) == \
        fa.FL_ERR_INVALID_ARG
    assert call(bias=_t((H, Nr, Nr)), mask=_t((Ns, Nr, 1, 1), dtype=fa.FL_F32)) == \
        fa.FL_ERR_INVALID_ARG
    odd = _t((Bt, Ns, Nr, H, c), strides=(Ns * Nr * H * c + 4, Nr * H * c, H * c, c, 1))
    assert call(q=odd) == fa.FL_ERR_ALIGNMENT


@fake_addresses
def test_diff_bwd_validation_before_device(lib):
    B, S, H, Hk = 2, 256, 4, 2
    r = ctypes.byref

    def args(Dv=128, do_shape=None):
        return [_t((2, B, S, H, 64)), _t((2, B, S, Hk, 64)), _t((B, S, Hk, Dv)), _t((2, B, H, S), fa.FL_F32),
                _t(do_shape or (B, S, H, Dv)), _t((2, B, S, H, 64)), _t((2, B, S, Hk, 64)), _t((B, S, Hk, Dv))]

    def call(a, desc, ws=0x40000, nbytes=1 << 30):
        return lib.fl_attn_diff_bwd(*[r(x) for x in a], r(desc), ws, nbytes, None)

    d = fa.make_desc(kind="diff", diff_lambda=0.8)
    n = ctypes.c_size_t()
    a = args()
    assert lib.fl_attn_diff_bwd_workspace_size(r(a[0]), r(a[1]), r(a[2]), r(d), r(n)) == fa.FL_OK
    assert n.value > 0 and n.value % 256 == 0
    # every failure below happens before any CUDA call
    assert call(args(), fa.make_desc(kind="standard")) == fa.FL_ERR_INVALID_ARG
    assert call(args(Dv=96), d) == fa.FL_ERR_UNSUPPORTED
    assert call(args(), fa.make_desc(kind="diff", mask="window", window=8)) == fa.FL_ERR_UNSUPPORTED
    assert call(args(), fa.make_desc(kind="diff", score_mod="softcap", softcap=20.0)) == fa.FL_ERR_UNSUPPORTED
    assert call(args(do_shape=(B, S, H, 64)), d) == fa.FL_ERR_INVALID_ARG
    assert call(args(), d, ws=0) == fa.FL_ERR_INVALID_ARG
    assert call(args(), d, ws=0x40010) == fa.FL_ERR_ALIGNMENT
    assert call(args(), d, nbytes=n.value - 1) == fa.FL_ERR_INVALID_ARG
    assert "workspace holds" in fa.fl_attn_last_error()
