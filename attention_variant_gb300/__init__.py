"""Python binding of the GB300 fused attention-variant forward (include/fl_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libflattn.so``.  There is no CPU fallback -- if the library
is missing, importing the binding's entry points raises.

The names mirror the C ABI: :func:`fl_attn_fwd`, :func:`fl_attn_tile_shape`,
:func:`fl_attn_status_string`, :func:`fl_attn_last_error`,
:func:`fl_attn_version`, :func:`fl_attn_decode_workspace_size`,
:func:`fl_attn_decode`, :func:`fl_attn_decode_static`, :func:`fl_attn_bwd`,
:func:`fl_attn_diff_bwd`.  Tensors are torch tensors on the current CUDA device
(PyTorch provides device memory and streams; nothing else).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libflattn.so")

# fl_status
FL_OK = 0
FL_ERR_INVALID_ARG = 1
FL_ERR_UNSUPPORTED = 2
FL_ERR_ALIGNMENT = 3
FL_ERR_CUDA = 4
FL_ERR_DEVICE_TIMEOUT = 5
FL_ERR_NO_DEVICE = 6
# fl_dtype
FL_BF16 = 0
FL_F32 = 1
# fl_kind
FL_KIND_STANDARD = 0
FL_KIND_DIFF = 1
FL_KIND_EVO_ROW = 2
FL_KIND_EVO_COL = 3
# fl_score_mod
FL_MOD_NONE = 0
FL_MOD_ALIBI = 1
FL_MOD_SOFTCAP = 2
FL_MOD_EXPR = 3
# fl_mask
FL_MASK_NONE = 0
FL_MASK_CAUSAL = 1
FL_MASK_WINDOW = 2
FL_MASK_PREFIX = 3
FL_MASK_DOC = 4
# fl_inject
FL_INJECT_NONE = 0
FL_INJECT_DROP_KV_LOAD = 1
FL_DEVERR_TIMEOUT = 0x1

MODS = {"none": FL_MOD_NONE, "vanilla": FL_MOD_NONE, "alibi": FL_MOD_ALIBI,
        "softcap": FL_MOD_SOFTCAP, "expr": FL_MOD_EXPR}
MASKS = {"none": FL_MASK_NONE, "causal": FL_MASK_CAUSAL, "window": FL_MASK_WINDOW,
         "prefix": FL_MASK_PREFIX, "doc": FL_MASK_DOC}
KINDS = {"standard": FL_KIND_STANDARD, "diff": FL_KIND_DIFF, "evo_row": FL_KIND_EVO_ROW,
         "evo_col": FL_KIND_EVO_COL}


class FlTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("sizes", ctypes.c_int64 * 5), ("strides", ctypes.c_int64 * 5)]


class FlDesc(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("score_mod", ctypes.c_int32), ("softcap", ctypes.c_float),
        ("mask", ctypes.c_int32), ("window", ctypes.c_int32), ("prefix", ctypes.c_int32),
        ("doc_offsets", ctypes.c_void_p), ("doc_stride", ctypes.c_int32),
        ("gqa_group", ctypes.c_int32), ("diff_lambda", ctypes.c_float), ("scale", ctypes.c_float),
        ("alibi_slopes", ctypes.c_void_p), ("debug_tile_counts", ctypes.c_void_p),
        ("error_word", ctypes.c_void_p), ("debug_inject", ctypes.c_int32),
        ("wait_timeout_us", ctypes.c_uint32), ("score_mod_expr", ctypes.c_char_p),
    ]


class FlDecodeDesc(ctypes.Structure):
    _fields_ = [
        ("score_mod", ctypes.c_int32), ("softcap", ctypes.c_float), ("causal", ctypes.c_int32),
        ("scale", ctypes.c_float), ("kv_lens", ctypes.c_void_p), ("max_kv_len", ctypes.c_int32),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int32),
        ("error_word", ctypes.c_void_p), ("wait_timeout_us", ctypes.c_uint32),
    ]


class FlAttnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{fl_attn_status_string(status)} ({detail})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: build it with `python -m attention_variant_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.fl_attn_fwd.restype = ctypes.c_int
    lib.fl_attn_fwd.argtypes = [P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor),
                                P(FlDesc), P(FlTensor), P(FlTensor), ctypes.c_void_p]
    lib.fl_attn_tile_shape.restype = ctypes.c_int
    lib.fl_attn_tile_shape.argtypes = [P(FlDesc), ctypes.c_int32, P(ctypes.c_int32),
                                       P(ctypes.c_int32)]
    lib.fl_attn_status_string.restype = ctypes.c_char_p
    lib.fl_attn_status_string.argtypes = [ctypes.c_int]
    lib.fl_attn_last_error.restype = ctypes.c_char_p
    lib.fl_attn_last_error.argtypes = []
    lib.fl_attn_version.restype = ctypes.c_int32
    lib.fl_attn_bwd_workspace_size.restype = ctypes.c_int
    lib.fl_attn_bwd_workspace_size.argtypes = [P(FlTensor), P(FlTensor), P(FlDesc),
                                               P(ctypes.c_size_t)]
    lib.fl_attn_bwd.restype = ctypes.c_int
    lib.fl_attn_bwd.argtypes = [P(FlTensor)] * 9 + [P(FlDesc), ctypes.c_void_p, ctypes.c_size_t,
                                                    ctypes.c_void_p]
    lib.fl_attn_diff_bwd_workspace_size.restype = ctypes.c_int
    lib.fl_attn_diff_bwd_workspace_size.argtypes = [P(FlTensor), P(FlTensor), P(FlTensor), P(FlDesc),
                                                    P(ctypes.c_size_t)]
    lib.fl_attn_diff_bwd.restype = ctypes.c_int
    lib.fl_attn_diff_bwd.argtypes = [P(FlTensor)] * 8 + [P(FlDesc), ctypes.c_void_p, ctypes.c_size_t,
                                                         ctypes.c_void_p]
    lib.fl_attn_evoformer.restype = ctypes.c_int
    lib.fl_attn_evoformer.argtypes = [P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor),
                                      P(FlDesc), P(FlTensor), P(FlTensor), P(FlTensor), ctypes.c_void_p]
    lib.fl_attn_score_expr_check.restype = ctypes.c_int
    lib.fl_attn_score_expr_check.argtypes = [ctypes.c_char_p, ctypes.c_int32]
    lib.fl_attn_decode_workspace_size.restype = ctypes.c_int
    lib.fl_attn_decode_workspace_size.argtypes = [P(FlTensor), P(FlTensor), P(FlDecodeDesc),
                                                  P(ctypes.c_size_t)]
    lib.fl_attn_decode_static.restype = ctypes.c_int
    lib.fl_attn_decode_static.argtypes = [P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor),
                                          P(FlTensor), P(FlDecodeDesc), ctypes.c_void_p]
    lib.fl_attn_decode.restype = ctypes.c_int
    lib.fl_attn_decode.argtypes = [P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor), P(FlTensor),
                                   P(FlDecodeDesc), ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.c_void_p]
    _lib = lib
    return lib


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FL_BF16
    if t.dtype == torch.float32:
        return FL_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def as_fl_tensor(t) -> FlTensor | None:
    """A torch tensor (or None) -> fl_tensor; no copy, no check."""
    if t is None:
        return None
    ft = FlTensor()
    ft.ptr = t.data_ptr()
    ft.dtype = _dtype_code(t)
    ft.ndim = t.dim()
    for d in range(t.dim()):
        ft.sizes[d] = t.shape[d]
        ft.strides[d] = t.stride(d)
    return ft


def make_desc(kind="standard", score_mod="none", softcap=20.0, mask="none", window=0, prefix=0,
              doc_offsets=None, gqa_group=0, diff_lambda=0.0, scale=0.0, alibi_slopes=None,
              debug_tile_counts=None, error_word=None, debug_inject=0,
              wait_timeout_us=0, score_expr=None) -> FlDesc:
    """Build an fl_attn_variant_desc; tensor arguments are device torch tensors.
    ``score_expr`` (a string in the grammar of include/fl_attn.h) selects
    FL_MOD_EXPR."""
    d = FlDesc()
    if score_expr is not None:
        score_mod = "expr"
        d.score_mod_expr = score_expr.encode()
    d.kind = KINDS[kind] if isinstance(kind, str) else int(kind)
    d.score_mod = MODS[score_mod] if isinstance(score_mod, str) else int(score_mod)
    d.softcap = float(softcap)
    d.mask = MASKS[mask] if isinstance(mask, str) else int(mask)
    d.window = int(window)
    d.prefix = int(prefix)
    if doc_offsets is not None:
        d.doc_offsets = doc_offsets.data_ptr()
        d.doc_stride = int(doc_offsets.shape[-1])
    d.gqa_group = int(gqa_group)
    d.diff_lambda = float(diff_lambda)
    d.scale = float(scale)
    d.alibi_slopes = alibi_slopes.data_ptr() if alibi_slopes is not None else None
    d.debug_tile_counts = debug_tile_counts.data_ptr() if debug_tile_counts is not None else None
    d.error_word = error_word.data_ptr() if error_word is not None else None
    d.debug_inject = int(debug_inject)
    d.wait_timeout_us = int(wait_timeout_us)
    return d


def _ref(x):
    return ctypes.byref(x) if x is not None else None


def fl_attn_bwd_workspace_size(q, k, desc: FlDesc) -> int:
    """Bytes of workspace fl_attn_bwd needs for these shapes."""
    lib = load_library()
    n = ctypes.c_size_t()
    st = lib.fl_attn_bwd_workspace_size(_ref(as_fl_tensor(q)), _ref(as_fl_tensor(k)), ctypes.byref(desc),
                                        ctypes.byref(n))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())
    return n.value


def fl_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, desc: FlDesc, workspace, stream=None) -> None:
    """Enqueue the backward (see include/fl_attn.h); workspace is a device torch
    tensor of at least fl_attn_bwd_workspace_size bytes."""
    lib = load_library()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    t = [as_fl_tensor(x) for x in (q, k, v, out, lse, dout, dq, dk, dv)]
    st = lib.fl_attn_bwd(*[_ref(x) for x in t], ctypes.byref(desc),
                         ctypes.c_void_p(workspace.data_ptr()),
                         workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_diff_bwd_workspace_size(q, k, v, desc: FlDesc) -> int:
    """Bytes of workspace fl_attn_diff_bwd needs for these shapes."""
    lib = load_library()
    n = ctypes.c_size_t()
    st = lib.fl_attn_diff_bwd_workspace_size(_ref(as_fl_tensor(q)), _ref(as_fl_tensor(k)), _ref(as_fl_tensor(v)),
                                             ctypes.byref(desc), ctypes.byref(n))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())
    return n.value


def fl_attn_diff_bwd(q, k, v, lse, dout, dq, dk, dv, desc: FlDesc, workspace, stream=None) -> None:
    """Enqueue the differential backward (see include/fl_attn.h); workspace is
    a device torch tensor of at least fl_attn_diff_bwd_workspace_size bytes."""
    lib = load_library()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    t = [as_fl_tensor(x) for x in (q, k, v, lse, dout, dq, dk, dv)]
    st = lib.fl_attn_diff_bwd(*[_ref(x) for x in t], ctypes.byref(desc),
                              ctypes.c_void_p(workspace.data_ptr()),
                              workspace.numel() * workspace.element_size(), ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_evoformer(q, k, v, out, lse, desc: FlDesc, bias=None, gate=None, msa_mask=None,
                      stream=None) -> None:
    """The Evoformer kinds over a batch of MSA stacks (5-D tensors) with an
    optional MSA mask (see include/fl_attn.h); raises FlAttnError."""
    lib = load_library()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    t = [as_fl_tensor(x) if x is not None else None for x in (q, k, v, out, lse, bias, gate, msa_mask)]
    st = lib.fl_attn_evoformer(_ref(t[0]), _ref(t[1]), _ref(t[2]), _ref(t[3]), _ref(t[4]),
                               ctypes.byref(desc), _ref(t[5]), _ref(t[6]), _ref(t[7]),
                               ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_score_expr_check(expr: str, compile=False) -> None:
    """Check a score_mod expression against the grammar; with ``compile`` true
    also run the runtime compilation of its forward kernel, with
    ``compile="backward"`` also that of its backward kernels (no GPU needed).
    Raises FlAttnError."""
    lib = load_library()
    level = 2 if compile == "backward" else int(bool(compile))
    st = lib.fl_attn_score_expr_check(expr.encode(), level)
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_fwd(q, k, v, out, lse=None, desc: FlDesc | None = None, bias=None, gate=None,
                stream=None) -> None:
    """Enqueue the fused forward on ``stream`` (default: torch's current stream).

    Raises :class:`FlAttnError` on a non-OK status.  See include/fl_attn.h for
    the layouts of each kind.
    """
    lib = load_library()
    if desc is None:
        desc = make_desc()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    tensors = [as_fl_tensor(x) for x in (q, k, v, out, lse, bias, gate)]
    st = lib.fl_attn_fwd(_ref(tensors[0]), _ref(tensors[1]), _ref(tensors[2]), _ref(tensors[3]),
                         _ref(tensors[4]), ctypes.byref(desc), _ref(tensors[5]),
                         _ref(tensors[6]), ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_tile_shape(desc: FlDesc, head_dim: int) -> tuple[int, int]:
    lib = load_library()
    bm, bn = ctypes.c_int32(), ctypes.c_int32()
    st = lib.fl_attn_tile_shape(ctypes.byref(desc), int(head_dim), ctypes.byref(bm),
                                ctypes.byref(bn))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())
    return bm.value, bn.value


def fl_attn_status_string(status: int) -> str:
    return load_library().fl_attn_status_string(int(status)).decode()


def fl_attn_last_error() -> str:
    return load_library().fl_attn_last_error().decode()


def fl_attn_version() -> int:
    return int(load_library().fl_attn_version())


def make_decode_desc(kv_lens, max_kv_len: int, *, score_mod="none", softcap=20.0, causal=True,
                     scale=0.0, block_table=None, error_word=None,
                     wait_timeout_us=0) -> FlDecodeDesc:
    """Build an fl_decode_desc; kv_lens and block_table are device int32 torch tensors."""
    d = FlDecodeDesc()
    d.score_mod = MODS[score_mod] if isinstance(score_mod, str) else int(score_mod)
    d.softcap = float(softcap)
    d.causal = 1 if causal else 0
    d.scale = float(scale)
    d.kv_lens = kv_lens.data_ptr()
    d.max_kv_len = int(max_kv_len)
    if block_table is not None:
        d.block_table = block_table.data_ptr()
        d.block_table_stride = int(block_table.stride(0))
    d.error_word = error_word.data_ptr() if error_word is not None else None
    d.wait_timeout_us = int(wait_timeout_us)
    d._keep = (kv_lens, block_table, error_word)
    return d


def fl_attn_decode_workspace_size(q, k_cache, desc: FlDecodeDesc) -> int:
    """Bytes of workspace fl_attn_decode needs for these shapes."""
    lib = load_library()
    n = ctypes.c_size_t()
    st = lib.fl_attn_decode_workspace_size(ctypes.byref(as_fl_tensor(q)),
                                           ctypes.byref(as_fl_tensor(k_cache)), ctypes.byref(desc),
                                           ctypes.byref(n))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())
    return n.value


def fl_attn_decode(q, k_cache, v_cache, out, lse, desc: FlDecodeDesc, workspace, stream=None) -> None:
    """Enqueue attention against a KV cache (see include/fl_attn.h); workspace is a
    device torch tensor of at least fl_attn_decode_workspace_size bytes."""
    lib = load_library()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    tensors = [as_fl_tensor(x) for x in (q, k_cache, v_cache, out, lse)]
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.fl_attn_decode(_ref(tensors[0]), _ref(tensors[1]), _ref(tensors[2]), _ref(tensors[3]),
                            _ref(tensors[4]), ctypes.byref(desc), ctypes.c_void_p(workspace.data_ptr()),
                            nbytes, ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())


def fl_attn_decode_static(q, k_cache, v_cache, out, lse, desc: FlDecodeDesc, stream=None) -> None:
    """fl_attn_decode with the library's own static scratch instead of a
    workspace: for callers that cannot allocate device memory.  Allocates
    nothing; calls that overlap on the GPU race (they share the scratch); the
    first call in a CUDA context (per device, and again after a device reset)
    sets up the scratch address, so make it before any stream capture."""
    lib = load_library()
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    tensors = [as_fl_tensor(x) for x in (q, k_cache, v_cache, out, lse)]
    st = lib.fl_attn_decode_static(_ref(tensors[0]), _ref(tensors[1]), _ref(tensors[2]),
                                   _ref(tensors[3]), _ref(tensors[4]), ctypes.byref(desc),
                                   ctypes.c_void_p(stream))
    if st != FL_OK:
        raise FlAttnError(st, fl_attn_last_error())

