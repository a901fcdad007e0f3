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
    assert _call(lib, _t((B, S, H, 128)), _t((B, S, H, 128)), _t((B, S, H, 128)),
                 _t((B, S, H, 128))) == fa.FL_ERR_UNSUPPORTED
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
    # a size-1 axis may carry any stride (torch often reports 1 there)
    q = _t((1, 256, 1, 64), strides=(1, 64, 1, 1))
    st = _call(lib, q, q, q, q)
    assert st not in (fa.FL_ERR_ALIGNMENT, fa.FL_ERR_INVALID_ARG), fa.fl_attn_last_error()


def test_tile_shape(lib):
    assert fa.fl_attn_tile_shape(fa.make_desc(), 64) == (128, 112)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="diff"), 64) == (128, 128)
    assert fa.fl_attn_tile_shape(fa.make_desc(kind="evo_row"), 32) == (128, 128)
    with pytest.raises(fa.FlAttnError):
        fa.fl_attn_tile_shape(fa.make_desc(), 48)
