"""GB300-native per-token-group FP8 activation quantization.

A thin ctypes binding over ``libtkq.so`` (C ABI in ``include/tkq.h``).  Every
step of the computation runs in the library's CUDA kernels; this module only
marshals pointers, sizes and the current CUDA stream, and allocates output
tensors with PyTorch.  There is no CPU fallback: if the library is missing or a
call fails, an exception is raised.

Low-level names mirror the C ABI (``tkq_per_token_cast``, ``tkq_swiglu_cast``,
``tkq_swiglu_cast_t``: raw device pointers, return the status code).  The
tensor-level helpers follow the call shape of the TileKernels quant API
(``per_token_cast(x, fmt='e4m3', num_per_channels=128) -> (out, out_sf)``,
"DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限", quick start).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

__all__ = [
    "TkqError", "library_path", "load_library", "tkq_per_token_cast", "tkq_swiglu_cast",
    "tkq_swiglu_cast_t", "tkq_swiglu_backward_cast", "tkq_status_string", "per_token_cast",
    "swiglu_forward_and_per_token_cast", "swiglu_backward_and_per_token_cast",
    "tkq_read_device_status", "tkq_selftest_wait_timeout", "FMT_E4M3", "FMT_E5M2", "GROUP",
    "tkq_per_channel_cast", "tkq_per_block_cast", "tkq_cast_back", "per_channel_cast",
    "per_block_cast", "cast_back", "OUT_F32", "OUT_BF16", "tkq_swiglu_cast_clamp",
    "tkq_swiglu_cast_t_clamp", "tkq_swiglu_cast_t_ex", "tkq_per_token_cast_f32", "tkq_swiglu_values", "swiglu_values",
    "use_checked_library", "tkq_checked_build", "tkq_read_check_address",
    "tkq_swiglu_backward_values", "swiglu_backward_values", "tkq_fp8_encode", "fp8_encode",
]

FMT_E4M3 = 0
FMT_E5M2 = 1
GROUP = 128
_FMTS = {"e4m3": FMT_E4M3, "e5m2": FMT_E5M2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libtkq.so")
# the access-checked test build of the same sources (see include/tkq.h)
_LIB_CHECKED_PATH = os.path.join(_HERE, "_lib", "libtkq_checked.so")
_lock = threading.RLock()
_lib = None          # the library every call of this module goes to
_opened = {}         # path -> loaded library


class TkqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {tkq_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libtkq.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(_LIB_PATH)
        return _lib


@contextlib.contextmanager
def use_checked_library():
    """Route this module's calls to the access-checked build libtkq_checked.so
    (built by ``_build.build(checked=True)``) inside the ``with`` block."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _open(_LIB_CHECKED_PATH)
    try:
        yield _lib
    finally:
        with _lock:
            _lib = prev


def _open(path):
    with _lock:
        if path in _opened:
            return _opened[path]
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        p, i64, i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.tkq_per_token_cast.argtypes = [p, p, p, i64, i64, i, i, p]
        lib.tkq_per_token_cast.restype = i
        lib.tkq_swiglu_cast.argtypes = [p, p, p, p, i64, i64, i, i, p]
        lib.tkq_swiglu_cast.restype = i
        lib.tkq_swiglu_cast_t.argtypes = [p, p, p, p, p, p, i64, i64, i, i, p]
        lib.tkq_swiglu_cast_t.restype = i
        lib.tkq_status_string.argtypes = [i]
        lib.tkq_status_string.restype = ctypes.c_char_p
        lib.tkq_version.argtypes = []
        lib.tkq_version.restype = i
        lib.tkq_swiglu_backward_cast.argtypes = [p, p, p, p, p, i64, i64, i, i, p]
        lib.tkq_swiglu_backward_cast.restype = i
        u = ctypes.c_uint
        lib.tkq_per_token_cast_ex.argtypes = [p, p, p, i64, i64, i, i, u, p]
        lib.tkq_per_token_cast_ex.restype = i
        lib.tkq_swiglu_cast_ex.argtypes = [p, p, p, p, i64, i64, i, i, u, p]
        lib.tkq_swiglu_cast_ex.restype = i
        lib.tkq_swiglu_backward_cast_ex.argtypes = [p, p, p, p, p, i64, i64, i, i, u, p]
        lib.tkq_swiglu_backward_cast_ex.restype = i
        lib.tkq_sf_bytes.argtypes = [i64, i64, u]
        lib.tkq_sf_bytes.restype = i64
        lib.tkq_read_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i]
        lib.tkq_read_device_status.restype = i
        lib.tkq_selftest_wait_timeout.argtypes = [i64, p]
        lib.tkq_selftest_wait_timeout.restype = i
        lib.tkq_per_channel_cast.argtypes = [p, p, p, i64, i64, i, i, i, p]
        lib.tkq_per_channel_cast.restype = i
        lib.tkq_per_block_cast.argtypes = [p, p, p, i64, i64, i, i, p]
        lib.tkq_per_block_cast.restype = i
        lib.tkq_cast_back.argtypes = [p, p, p, i64, i64, i, i, i, i, p]
        lib.tkq_cast_back.restype = i
        f32 = ctypes.c_float
        lib.tkq_swiglu_cast_clamp.argtypes = [p, p, p, p, i64, i64, i, i, u, f32, p, p]
        lib.tkq_swiglu_cast_clamp.restype = i
        lib.tkq_swiglu_cast_t_clamp.argtypes = [p, p, p, p, p, p, i64, i64, i, i, u, f32, p, p]
        lib.tkq_swiglu_cast_t_clamp.restype = i
        lib.tkq_swiglu_cast_t_ex.argtypes = [p, p, p, p, p, p, i64, i64, i, i, u, p]
        lib.tkq_swiglu_cast_t_ex.restype = i
        lib.tkq_per_token_cast_f32.argtypes = [p, p, p, i64, i64, i, i, u, p]
        lib.tkq_per_token_cast_f32.restype = i
        lib.tkq_swiglu_values.argtypes = [p, p, p, i64, i64, p]
        lib.tkq_swiglu_values.restype = i
        lib.tkq_swiglu_backward_values.argtypes = [p, p, p, p, i64, i64, p]
        lib.tkq_swiglu_backward_values.restype = i
        lib.tkq_fp8_encode.argtypes = [p, p, i64, i, p]
        lib.tkq_fp8_encode.restype = i
        lib.tkq_checked_build.argtypes = []
        lib.tkq_checked_build.restype = i
        lib.tkq_read_check_address.argtypes = [ctypes.POINTER(ctypes.c_uint64), i]
        lib.tkq_read_check_address.restype = i
        _opened[path] = lib
        return lib


DEVICE_TIMEOUT = 1
ERR_TIMEOUT = 7    # tkq_read_device_status: the status word holds DEVICE_TIMEOUT
DEVICE_OUT_OF_BOUNDS = 2


def tkq_checked_build() -> bool:
    return bool((_lib or load_library()).tkq_checked_build())


def tkq_read_check_address(clear: bool = False) -> int:
    """Synchronize the current device and return the first address an access
    check refused (bit 63 set for a store; 0 if none, and always 0 in the
    release build)."""
    v = ctypes.c_uint64(0)
    st = (_lib or load_library()).tkq_read_check_address(ctypes.byref(v), 1 if clear else 0)
    if st:
        raise TkqError(st, "tkq_read_check_address")
    return int(v.value)


def tkq_read_device_status(clear: bool = False) -> int:
    """Synchronize the current device and return its status word (bit
    DEVICE_TIMEOUT: a bounded wait inside a kernel gave up; the C call then
    returns ERR_TIMEOUT, which here is the word's bit, not an exception)."""
    v = ctypes.c_uint32(0)
    st = (_lib or load_library()).tkq_read_device_status(ctypes.byref(v), 1 if clear else 0)
    if st and st != ERR_TIMEOUT:
        raise TkqError(st, "tkq_read_device_status")
    return int(v.value)


def tkq_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return (_lib or load_library()).tkq_selftest_wait_timeout(int(limit_ns), stream)


def tkq_status_string(status: int) -> str:
    return (_lib or load_library()).tkq_status_string(int(status)).decode()


# ---------------------------------------------------------------------------
# C-ABI mirrors: raw device pointers (ints or None), sizes, stream handle.
# ---------------------------------------------------------------------------

def tkq_per_token_cast(x, out, sf, T, C, group=GROUP, fmt=FMT_E4M3, stream=None) -> int:
    return (_lib or load_library()).tkq_per_token_cast(x, out, sf, T, C, group, fmt, stream)


def tkq_swiglu_cast(x, w, out, sf, T, H, group=GROUP, fmt=FMT_E4M3, stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast(x, w, out, sf, T, H, group, fmt, stream)


def tkq_swiglu_cast_t(x, w, out, sf, out_t, sf_t, T, H, group=GROUP, fmt=FMT_E4M3,
                      stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast_t(x, w, out, sf, out_t, sf_t, T, H, group, fmt, stream)


def tkq_swiglu_backward_cast(x, dy, w, out, sf, T, H, group=GROUP, fmt=FMT_E4M3,
                             stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_backward_cast(x, dy, w, out, sf, T, H, group, fmt, stream)


def tkq_per_token_cast_f32(x, out, sf, T, C, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                           stream=None) -> int:
    return (_lib or load_library()).tkq_per_token_cast_f32(x, out, sf, T, C, group, fmt, sf_flags, stream)


def tkq_swiglu_values(x, w, y, T, H, stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_values(x, w, y, T, H, stream)


def tkq_fp8_encode(x, out, n, fmt=FMT_E4M3, stream=None) -> int:
    return (_lib or load_library()).tkq_fp8_encode(x, out, n, fmt, stream)


def tkq_swiglu_backward_values(x, dy, w, y, T, H, stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_backward_values(x, dy, w, y, T, H, stream)


def tkq_swiglu_cast_clamp(x, w, out, sf, T, H, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                          clamp_value=0.0, clamp_count=None, stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast_clamp(x, w, out, sf, T, H, group, fmt, sf_flags,
                                                clamp_value, clamp_count, stream)


def tkq_swiglu_cast_t_clamp(x, w, out, sf, out_t, sf_t, T, H, group=GROUP, fmt=FMT_E4M3,
                            sf_flags=0, clamp_value=0.0, clamp_count=None, stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast_t_clamp(x, w, out, sf, out_t, sf_t, T, H, group,
                                                            fmt, sf_flags, clamp_value, clamp_count,
                                                            stream)


def tkq_swiglu_cast_t_ex(x, w, out, sf, out_t, sf_t, T, H, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                         stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast_t_ex(x, w, out, sf, out_t, sf_t, T, H, group,
                                                         fmt, sf_flags, stream)


def tkq_per_channel_cast(x, out, sf, T, C, group=GROUP, fmt=FMT_E4M3, transpose=0,
                         stream=None) -> int:
    return (_lib or load_library()).tkq_per_channel_cast(x, out, sf, T, C, group, fmt, int(transpose),
                                               stream)


def tkq_per_block_cast(x, out, sf, T, C, block=GROUP, fmt=FMT_E4M3, stream=None) -> int:
    return (_lib or load_library()).tkq_per_block_cast(x, out, sf, T, C, block, fmt, stream)


OUT_F32 = 0
OUT_BF16 = 1


def tkq_cast_back(codes, sf, out, T, C, group_rows=1, group_cols=GROUP, fmt=FMT_E4M3,
                  out_dtype=OUT_F32, stream=None) -> int:
    return (_lib or load_library()).tkq_cast_back(codes, sf, out, T, C, group_rows, group_cols, fmt,
                                        out_dtype, stream)


SF_ROUND_POW2 = 1
SF_UE8M0_PACKED = 2
SF_COL_MAJOR = 4
Q_RECIPROCAL = 8   # plain casts: codes of x * fl32(1/s) instead of fl32(x/s)


def tkq_sf_bytes(T, groups_per_row, sf_flags=0) -> int:
    return (_lib or load_library()).tkq_sf_bytes(T, groups_per_row, sf_flags)


def tkq_per_token_cast_ex(x, out, sf, T, C, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                          stream=None) -> int:
    return (_lib or load_library()).tkq_per_token_cast_ex(x, out, sf, T, C, group, fmt, sf_flags, stream)


def tkq_swiglu_cast_ex(x, w, out, sf, T, H, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                       stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_cast_ex(x, w, out, sf, T, H, group, fmt, sf_flags, stream)


def tkq_swiglu_backward_cast_ex(x, dy, w, out, sf, T, H, group=GROUP, fmt=FMT_E4M3, sf_flags=0,
                                stream=None) -> int:
    return (_lib or load_library()).tkq_swiglu_backward_cast_ex(x, dy, w, out, sf, T, H, group, fmt,
                                                      sf_flags, stream)


def _sf_shape(T: int, groups_per_row: int, sf_flags: int):
    """Shape and element type of the scales in the layout `sf_flags` selects:
    fp32 [T, G], fp32 [G, T4], int32 [T, W] or int32 [W, T4] (T4 = T rounded
    up to 4, W = G / 4 rounded up)."""
    T4 = (T + 3) // 4 * 4
    W = (groups_per_row + 3) // 4
    if sf_flags & SF_UE8M0_PACKED:
        return ((W, T4) if sf_flags & SF_COL_MAJOR else (T, W)), "int32"
    return ((groups_per_row, T4) if sf_flags & SF_COL_MAJOR else (T, groups_per_row)), "float32"


def sf_tensor(T: int, groups_per_row: int, sf_flags: int, device):
    """An empty scale tensor shaped for the layout `sf_flags` selects:
    fp32 [T, G], fp32 [G, T4], int32 [T, W] or int32 [W, T4]."""
    import torch
    shape, dt = _sf_shape(T, groups_per_row, sf_flags)
    return torch.empty(shape, dtype=getattr(torch, dt), device=device)


# ---------------------------------------------------------------------------
# Tensor-level helpers (PyTorch supplies device memory and the stream).
# ---------------------------------------------------------------------------

def _fmt_code(fmt) -> int:
    if isinstance(fmt, str):
        if fmt not in _FMTS:
            raise ValueError(f"unknown fmt {fmt!r}: expected 'e4m3' or 'e5m2'")
        return _FMTS[fmt]
    return int(fmt)


def _fp8_dtype(fmt_code: int):
    import torch
    return torch.float8_e4m3fn if fmt_code == FMT_E4M3 else torch.float8_e5m2


def _check_input(x, name="x", allow_f32=False):
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    ok = (torch.bfloat16, torch.float32) if allow_f32 else (torch.bfloat16,)
    if x.dtype not in ok or x.dim() != 2 or not x.is_contiguous():
        raise TypeError(f"{name} must be a contiguous 2-D "
                        + ("bfloat16 or float32" if allow_f32 else "bfloat16") + " tensor")


def _check_out(t, name, x, nbytes, itemsize=None, dtype=None):
    """A caller-supplied output buffer: a contiguous CUDA tensor on x's device
    of at least `nbytes` bytes (the kernels write exactly the bytes the call's
    shape and layout give, so a smaller buffer would be written past its end).
    `itemsize` / `dtype` pin the element size or type where the layout fixes
    them; scale buffers of any element type are accepted by size."""
    import torch
    if not isinstance(t, torch.Tensor) or t.device != x.device or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor on x's device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    if itemsize is not None and t.element_size() != itemsize:
        raise TypeError(f"{name} must have {itemsize}-byte elements")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes; "
                         f"the call writes {nbytes}")


def _check_sf_out(t, name, x, rows, groups_per_row, sf_flags):
    shape, _ = _sf_shape(rows, groups_per_row, sf_flags)
    _check_out(t, name, x, 4 * shape[0] * shape[1])


def _stream_handle(dev):
    """The current stream of `dev` as an int (ctypes passes it as void*).
    torch's raw-stream query avoids building a Stream object per call; the
    public call is used where that query does not exist."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(dev.index if dev.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


_NO_CONTEXT = contextlib.nullcontext()


def _device_ctx(dev):
    """The launch must happen on the tensors' device: switch only if it is not
    the current one (entering torch.cuda.device costs more than the launch)."""
    import torch
    if dev.index is None or dev.index == torch.cuda.current_device():
        return _NO_CONTEXT
    return torch.cuda.device(dev)


def _sf_flags(round_sf: bool, use_packed_ue8m0: bool, use_tma_aligned_col_major_sf: bool) -> int:
    """The TileKernels cast-config options ("DeepSeek开源TileKernels..." §3.1) as
    the C ABI's TKQ_SF_* flags."""
    return ((SF_ROUND_POW2 if round_sf else 0) | (SF_UE8M0_PACKED if use_packed_ue8m0 else 0)
            | (SF_COL_MAJOR if use_tma_aligned_col_major_sf else 0))


def _check_weights(topk_weights, T, x):
    import torch
    if topk_weights is not None:
        if (topk_weights.dtype != torch.float32 or topk_weights.numel() != T
                or not topk_weights.is_contiguous() or topk_weights.device != x.device):
            raise TypeError("topk_weights must be a contiguous fp32 tensor of T elements on x's device")


def per_token_cast(x, fmt="e4m3", num_per_channels: int = GROUP, out=None, out_sf=None,
                   round_sf: bool = False, use_packed_ue8m0: bool = False,
                   use_tma_aligned_col_major_sf: bool = False, use_sf_inv: bool = False):
    """bf16 or fp32 [T, C] -> (FP8 codes [T, C], scales).  Scales are fp32
    [T, C/128] unless a scale-layout option is set (see ``sf_tensor`` for the
    shapes).  Codes are those of the exact quotient x / s, or with
    ``use_sf_inv`` those of the product x * fl32(1 / s) (TKQ_Q_RECIPROCAL)."""
    import torch
    _check_input(x, allow_f32=True)
    f = _fmt_code(fmt)
    T, C = x.shape
    flags = _sf_flags(round_sf, use_packed_ue8m0, use_tma_aligned_col_major_sf)
    if use_sf_inv:
        flags |= Q_RECIPROCAL
    G = C // max(num_per_channels, 1)
    if out is None:
        out = torch.empty((T, C), dtype=_fp8_dtype(f), device=x.device)
    else:
        _check_out(out, "out", x, T * C, itemsize=1)
    if out_sf is None:
        out_sf = sf_tensor(T, G, flags, x.device)
    else:
        _check_sf_out(out_sf, "out_sf", x, T, G, flags)
    with _device_ctx(x.device):
        call = tkq_per_token_cast_f32 if x.dtype == torch.float32 else tkq_per_token_cast_ex
        st = call(_ptr(x), _ptr(out), _ptr(out_sf), T, C, num_per_channels, f, flags,
                  _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_per_token_cast")
    return out, out_sf


def swiglu_forward_and_per_token_cast(x, fmt="e4m3", num_per_channels: int = GROUP,
                                      topk_weights=None, with_transpose: bool = False,
                                      out=None, out_sf=None, out_t=None, out_sf_t=None,
                                      round_sf: bool = False, use_packed_ue8m0: bool = False,
                                      use_tma_aligned_col_major_sf: bool = False,
                                      use_clamp: bool = False, swiglu_clamp_value=None,
                                      clamp_count=None):
    """bf16 [T, 2H] (gate | up) -> (codes [T, H], scales [T, H/128]) and, with
    ``with_transpose``, also (codes_t [H, T], scales_t [H, T/128]).
    ``topk_weights``: optional fp32 [T] routing weight per row.  The scale-layout
    options apply to the row scales and, with ``with_transpose``, to the column
    scales as an [H, T/128] matrix (see ``sf_tensor`` for the shapes).  Codes
    are those of the product y * fl32(1 / s) (the TileKernels sf_inv reading).
    ``use_clamp``: clamp the gate to <= swiglu_clamp_value and the up projection
    to [-swiglu_clamp_value, swiglu_clamp_value] before the SwiGLU; the number of
    changed values is added to ``clamp_count`` (a zeroed int64 CUDA tensor of one
    element) when given."""
    import torch
    _check_input(x)
    clamp = None
    if use_clamp:
        if swiglu_clamp_value is None:
            raise ValueError("use_clamp needs swiglu_clamp_value")
        clamp = float(swiglu_clamp_value)
        if clamp_count is not None and (clamp_count.dtype != torch.int64 or clamp_count.numel() != 1
                                        or clamp_count.device != x.device):
            raise TypeError("clamp_count must be a one-element int64 tensor on x's device")
    elif clamp_count is not None:
        raise ValueError("clamp_count needs use_clamp")
    f = _fmt_code(fmt)
    T, H2 = x.shape
    if H2 % 2:
        raise ValueError("x must have an even number of columns (gate | up)")
    H = H2 // 2
    g = max(num_per_channels, 1)
    _check_weights(topk_weights, T, x)
    flags = _sf_flags(round_sf, use_packed_ue8m0, use_tma_aligned_col_major_sf)
    if out is None:
        out = torch.empty((T, H), dtype=_fp8_dtype(f), device=x.device)
    else:
        _check_out(out, "out", x, T * H, itemsize=1)
    if out_sf is None:
        out_sf = sf_tensor(T, H // g, flags, x.device)
    else:
        _check_sf_out(out_sf, "out_sf", x, T, H // g, flags)
    with _device_ctx(x.device):
        stream = _stream_handle(x.device)
        if not with_transpose:
            if clamp is None:
                st = tkq_swiglu_cast_ex(_ptr(x), _ptr(topk_weights), _ptr(out), _ptr(out_sf), T,
                                        H, num_per_channels, f, flags, stream)
            else:
                st = tkq_swiglu_cast_clamp(_ptr(x), _ptr(topk_weights), _ptr(out), _ptr(out_sf),
                                           T, H, num_per_channels, f, flags, clamp,
                                           _ptr(clamp_count), stream)
            if st:
                raise TkqError(st, "tkq_swiglu_cast")
            return out, out_sf
        if out_t is None:
            out_t = torch.empty((H, T), dtype=_fp8_dtype(f), device=x.device)
        else:
            _check_out(out_t, "out_t", x, H * T, itemsize=1)
        if out_sf_t is None:
            out_sf_t = sf_tensor(H, T // g, flags, x.device)
        else:
            _check_sf_out(out_sf_t, "out_sf_t", x, H, T // g, flags)
        if clamp is None:
            st = tkq_swiglu_cast_t_ex(_ptr(x), _ptr(topk_weights), _ptr(out), _ptr(out_sf),
                                      _ptr(out_t), _ptr(out_sf_t), T, H, num_per_channels, f,
                                      flags, stream)
        else:
            st = tkq_swiglu_cast_t_clamp(_ptr(x), _ptr(topk_weights), _ptr(out), _ptr(out_sf),
                                         _ptr(out_t), _ptr(out_sf_t), T, H, num_per_channels, f,
                                         flags, clamp, _ptr(clamp_count), stream)
        if st:
            raise TkqError(st, "tkq_swiglu_cast_t")
        return out, out_sf, out_t, out_sf_t


def swiglu_backward_and_per_token_cast(x, dy, fmt="e4m3", num_per_channels: int = GROUP,
                                       topk_weights=None, out=None, out_sf=None,
                                       round_sf: bool = False, use_packed_ue8m0: bool = False,
                                       use_tma_aligned_col_major_sf: bool = False):
    """Gradients of y = silu(gate) * up [* w] from dy, cast per token.
    x: bf16 [T, 2H] (gate | up); dy: bf16 [T, H] -> (codes [T, 2H] of [dg | du],
    scales [T, 2H/128] or the chosen scale layout); codes of the products by
    fl32(1 / s), like the forward cast."""
    import torch
    _check_input(x)
    _check_input(dy, "dy")
    f = _fmt_code(fmt)
    T, H2 = x.shape
    H = H2 // 2
    if H2 % 2 or tuple(dy.shape) != (T, H) or dy.device != x.device:
        raise ValueError("dy must be [T, H] for x [T, 2H], on the same device")
    _check_weights(topk_weights, T, x)
    g = max(num_per_channels, 1)
    flags = _sf_flags(round_sf, use_packed_ue8m0, use_tma_aligned_col_major_sf)
    if out is None:
        out = torch.empty((T, 2 * H), dtype=_fp8_dtype(f), device=x.device)
    else:
        _check_out(out, "out", x, T * 2 * H, itemsize=1)
    if out_sf is None:
        out_sf = sf_tensor(T, 2 * H // g, flags, x.device)
    else:
        _check_sf_out(out_sf, "out_sf", x, T, 2 * H // g, flags)
    with _device_ctx(x.device):
        st = tkq_swiglu_backward_cast_ex(_ptr(x), _ptr(dy), _ptr(topk_weights), _ptr(out),
                                         _ptr(out_sf), T, H, num_per_channels, f, flags,
                                         _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_swiglu_backward_cast")
    return out, out_sf


def per_channel_cast(x, fmt="e4m3", num_per_channels: int = GROUP, transpose: bool = False,
                     out=None, out_sf=None):
    """bf16 [T, C] -> codes and scales of groups of 128 tokens per channel:
    (codes [T, C], scales [T/128, C]), or with ``transpose`` the column-major
    copy (codes [C, T], scales [C, T/128]).  T must be a multiple of 128."""
    import torch
    _check_input(x)
    f = _fmt_code(fmt)
    T, C = x.shape
    g = max(num_per_channels, 1)
    if out is None:
        out = torch.empty((C, T) if transpose else (T, C), dtype=_fp8_dtype(f), device=x.device)
    else:
        _check_out(out, "out", x, T * C, itemsize=1)
    if out_sf is None:
        out_sf = torch.empty((C, T // g) if transpose else (T // g, C), dtype=torch.float32,
                             device=x.device)
    else:
        _check_out(out_sf, "out_sf", x, 4 * C * (T // g))
    with _device_ctx(x.device):
        st = tkq_per_channel_cast(_ptr(x), _ptr(out), _ptr(out_sf), T, C, num_per_channels, f,
                                  int(transpose), _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_per_channel_cast")
    return out, out_sf


def per_block_cast(x, fmt="e4m3", block_size: int = GROUP, out=None, out_sf=None):
    """bf16 [T, C] -> (codes [T, C], scales [ceil(T/128), C/128]), one scale per
    128 x 128 block."""
    import torch
    _check_input(x)
    f = _fmt_code(fmt)
    T, C = x.shape
    b = max(block_size, 1)
    if out is None:
        out = torch.empty((T, C), dtype=_fp8_dtype(f), device=x.device)
    else:
        _check_out(out, "out", x, T * C, itemsize=1)
    if out_sf is None:
        out_sf = torch.empty(((T + b - 1) // b, C // b), dtype=torch.float32, device=x.device)
    else:
        _check_out(out_sf, "out_sf", x, 4 * ((T + b - 1) // b) * (C // b))
    with _device_ctx(x.device):
        st = tkq_per_block_cast(_ptr(x), _ptr(out), _ptr(out_sf), T, C, block_size, f,
                                _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_per_block_cast")
    return out, out_sf


def cast_back(x, sf, fmt=None, group_size=(1, GROUP), out_dtype=None, out=None):
    """FP8 codes [T, C] and fp32 scales -> decode(code) * scale as fp32 (default)
    or bf16.  ``group_size`` = (rows, cols) of one scale group: (1, 128)
    per-token, (128, 1) per-channel, (128, 128) per-block.  ``fmt`` defaults to
    the codes' dtype (float8_e4m3fn or float8_e5m2; uint8 codes need fmt)."""
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 2 or not x.is_contiguous():
        raise TypeError("x must be a contiguous 2-D CUDA tensor of FP8 codes")
    if x.element_size() != 1:
        raise TypeError("x must hold one-byte FP8 codes")
    if fmt is None:
        if x.dtype == torch.float8_e4m3fn:
            fmt = "e4m3"
        elif x.dtype == torch.float8_e5m2:
            fmt = "e5m2"
        else:
            raise ValueError("fmt is required for codes that are not an FP8 dtype")
    f = _fmt_code(fmt)
    if (not isinstance(sf, torch.Tensor) or sf.dtype != torch.float32 or not sf.is_contiguous()
            or sf.device != x.device):
        raise TypeError("sf must be a contiguous fp32 tensor on the codes' device")
    gr, gc = group_size
    T, C = x.shape
    if (-(-T // max(gr, 1)), C // max(gc, 1)) != tuple(sf.shape[-2:]) or sf.dim() != 2:
        raise ValueError(f"sf must have shape [ceil(T/{gr}), C/{gc}]")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((T, C), dtype=out_dtype, device=x.device)
    else:
        _check_out(out, "out", x, T * C * (4 if out_dtype == torch.float32 else 2),
                   dtype=out_dtype)
    code = OUT_F32 if out_dtype == torch.float32 else OUT_BF16
    with _device_ctx(x.device):
        st = tkq_cast_back(_ptr(x), _ptr(sf), _ptr(out), T, C, gr, gc, f, code,
                           _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_cast_back")
    return out


def swiglu_values(x, topk_weights=None):
    """Diagnostic: the fp32 SwiGLU values [T, H] exactly as the SwiGLU casts
    compute them before quantizing (x: bf16 [T, 2H] gate | up)."""
    import torch
    _check_input(x)
    T, H2 = x.shape
    if H2 % 2:
        raise ValueError("x must have an even number of columns (gate | up)")
    _check_weights(topk_weights, T, x)
    y = torch.empty((T, H2 // 2), dtype=torch.float32, device=x.device)
    with _device_ctx(x.device):
        st = tkq_swiglu_values(_ptr(x), _ptr(topk_weights), _ptr(y), T, H2 // 2,
                               _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_swiglu_values")
    return y


def swiglu_backward_values(x, dy, topk_weights=None):
    """Diagnostic: the fp32 gradients [dg | du] ([T, 2H]) exactly as the SwiGLU
    backward cast computes them before quantizing (x: bf16 [T, 2H] gate | up,
    dy: bf16 [T, H])."""
    import torch
    _check_input(x)
    _check_input(dy, "dy")
    T, H2 = x.shape
    H = H2 // 2
    if H2 % 2 or tuple(dy.shape) != (T, H) or dy.device != x.device:
        raise ValueError("dy must be [T, H] for x [T, 2H], on the same device")
    _check_weights(topk_weights, T, x)
    y = torch.empty((T, H2), dtype=torch.float32, device=x.device)
    with _device_ctx(x.device):
        st = tkq_swiglu_backward_values(_ptr(x), _ptr(dy), _ptr(topk_weights), _ptr(y), T, H,
                                        _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_swiglu_backward_values")
    return y


def fp8_encode(x, fmt="e4m3"):
    """Diagnostic: the FP8 codes (uint8, same shape) of an fp32 CUDA tensor,
    unscaled, by the conversion every cast ends with."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous fp32 CUDA tensor")
    f = _fmt_code(fmt)
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    with _device_ctx(x.device):
        st = tkq_fp8_encode(_ptr(x), _ptr(out), x.numel(), f, _stream_handle(x.device))
    if st:
        raise TkqError(st, "tkq_fp8_encode")
    return out
