"""CPU oracle for per-token-group FP8 activation quantization.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only code allowed to import
this package.  The product path (the CUDA library and its Python binding)
never imports, links or calls it, and this package never imports the product.

The arithmetic lives in ``tkq_oracle.c`` (plain single-threaded C, binary32
steps in round-to-nearest-even, compiled without FMA contraction); this module
only builds it with gcc and marshals numpy arrays through ctypes.  bf16 inputs
are passed as ``uint16`` bit patterns; codes come back as ``uint8``.

Sources: the TileKernels walkthrough "DeepSeek开源TileKernels：用Python写的GPU
算子逼近硬件性能上限" (itsolotime.com) §3.1-§3.3, the operator table of
"TileKernels 与 DeepGEMM 的分界线" (chatdocs.ruinique.com) §2, and the quant/
section of "刚刚！DeepSeek开源高性能GPU算子库TileKernels" (info.datadowell.com).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
FMT = {"e4m3": E4M3, "e5m2": E5M2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tkq_oracle.c")
_LIB = os.path.join(_HERE, "libtkq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``tkq_oracle.c`` into ``libtkq_oracle.so`` next to it."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "tkq_oracle.h"))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def build_variant(src_text: str, out_dir: str) -> str:
    """Compile a modified copy of the oracle source (used by the mutation tests
    that show the pins reject a planted mistake) and return the library path."""
    src = os.path.join(out_dir, "tkq_oracle.c")
    with open(src, "w") as f:
        f.write(src_text)
    hdr = os.path.join(out_dir, "tkq_oracle.h")
    with open(os.path.join(_HERE, "tkq_oracle.h")) as f, open(hdr, "w") as g:
        g.write(f.read())
    lib = os.path.join(out_dir, "libtkq_oracle_variant.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-o", lib, src, "-lm"], check=True)
    return lib


class use_library:
    """Context manager: route every call of this module to another build of the
    oracle (a planted-mistake variant) and restore the real one afterwards."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self.saved = _lib
            _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _configure(ctypes.CDLL(_LIB))
    return _lib


def _configure(lib):
    """Declare the C signatures on a freshly loaded oracle library."""
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    i = ctypes.c_int
    lib.ora_fp8_max.argtypes = [i]
    lib.ora_fp8_max.restype = ctypes.c_double
    lib.ora_fp8_decode.argtypes = [ctypes.c_uint8, i]
    lib.ora_fp8_decode.restype = ctypes.c_double
    lib.ora_fp8_encode.argtypes = [ctypes.c_float, i]
    lib.ora_fp8_encode.restype = ctypes.c_uint8
    lib.ora_fp8_encode_array.argtypes = [p, i64, i, p]
    lib.ora_fp8_encode_array.restype = ctypes.c_int
    lib.ora_group_scale.argtypes = [ctypes.c_float, i]
    lib.ora_group_scale.restype = ctypes.c_float
    lib.ora_per_token_cast.argtypes = [p, i64, i64, i64, i, p, p]
    lib.ora_cast_rows_f32.argtypes = [p, i64, i64, i64, i, p, p]
    lib.ora_cast_cols_f32.argtypes = [p, i64, i64, i64, i, p, p]
    lib.ora_swiglu_values.argtypes = [p, p, i64, i64, p]
    lib.ora_swiglu_cast.argtypes = [p, p, i64, i64, i64, i, p, p]
    lib.ora_swiglu_cast_t.argtypes = [p, p, i64, i64, i64, i, p, p, p, p]
    lib.ora_pow2_ceil.argtypes = [ctypes.c_float]
    lib.ora_pow2_ceil.restype = ctypes.c_float
    lib.ora_sf_bytes.argtypes = [i64, i64, i]
    lib.ora_sf_bytes.restype = i64
    lib.ora_cast_rows_f32_ex.argtypes = [p, i64, i64, i64, i, i, p, p]
    lib.ora_cast_rows_f32_ex.restype = ctypes.c_int
    lib.ora_per_channel_cast.argtypes = [p, i64, i64, i64, i, i, p, p]
    lib.ora_per_channel_cast.restype = ctypes.c_int
    lib.ora_per_block_cast.argtypes = [p, i64, i64, i64, i, p, p]
    lib.ora_per_block_cast.restype = ctypes.c_int
    lib.ora_cast_back.argtypes = [p, p, i64, i64, i64, i64, i, p]
    lib.ora_cast_back.restype = ctypes.c_int
    lib.ora_swiglu_backward_values.argtypes = [p, p, p, i64, i64, p]
    lib.ora_swiglu_backward_cast.argtypes = [p, p, p, i64, i64, i64, i, p, p]
    lib.ora_swiglu_values_clamp.argtypes = [p, p, i64, i64, p, p, p]
    lib.ora_swiglu_cast_clamp.argtypes = [p, p, i64, i64, i64, i, p, p, p, p]
    lib.ora_swiglu_cast_t_clamp.argtypes = [p, p, i64, i64, i64, i, p, p, p, p, p, p]
    for f in ("ora_swiglu_values_clamp", "ora_swiglu_cast_clamp", "ora_swiglu_cast_t_clamp",
              "ora_per_token_cast", "ora_cast_rows_f32", "ora_cast_cols_f32",
              "ora_swiglu_values", "ora_swiglu_cast", "ora_swiglu_cast_t",
              "ora_swiglu_backward_values", "ora_swiglu_backward_cast"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _fmt(fmt) -> int:
    return FMT[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


# --------------------------------------------------------------------------
# scalar codec
# --------------------------------------------------------------------------

def fp8_max(fmt) -> float:
    return _load().ora_fp8_max(_fmt(fmt))


def fp8_decode(code: int, fmt) -> float:
    return _load().ora_fp8_decode(int(code) & 0xFF, _fmt(fmt))


def fp8_encode(v: float, fmt) -> int:
    return int(_load().ora_fp8_encode(float(np.float32(v)), _fmt(fmt)))


def fp8_encode_array(v: np.ndarray, fmt, out: np.ndarray | None = None) -> np.ndarray:
    """Encode every binary32 value of ``v`` (into ``out`` if given: uint8,
    contiguous, the size of ``v``)."""
    lib = _load()
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    if out is None:
        out = np.empty(flat.shape, np.uint8)
    elif out.dtype != np.uint8 or out.size != flat.size or not out.flags.c_contiguous:
        raise ValueError("out must be a contiguous uint8 array of the input's size")
    _check(lib.ora_fp8_encode_array(_ptr(flat), flat.size, _fmt(fmt), _ptr(out)), "encode_array")
    return out.reshape(np.shape(v))


def group_scale(amax: float, fmt) -> np.float32:
    return np.float32(_load().ora_group_scale(float(np.float32(amax)), _fmt(fmt)))


# --------------------------------------------------------------------------
# casts (rows are independent; ``threads`` splits row ranges across threads,
# ctypes releases the GIL during each call)
# --------------------------------------------------------------------------

def _row_parallel(T: int, threads: int, body, align: int = 1):
    threads = max(1, min(int(threads), max(1, T // max(align, 1))))
    if threads == 1:
        body(0, T)
        return
    per = -(-T // threads)
    per = -(-per // align) * align
    errs = []

    def run(a, b):
        try:
            body(a, b)
        except Exception as e:  # pragma: no cover - surfaced below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(a, min(T, a + per)))
          for a in range(0, T, per)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errs:
        raise errs[0]


def per_token_cast(x_bits: np.ndarray, fmt="e4m3", group: int = 128, threads: int = 1):
    """x_bits: uint16 [T, C] (bf16 bits) -> (codes uint8 [T, C], sf float32 [T, C/group])."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, C = x_bits.shape
    if group <= 0 or C % group:
        raise ValueError("group must divide C")
    out = np.empty((T, C), np.uint8)
    sf = np.empty((T, C // group), np.float32)
    f = _fmt(fmt)

    def body(a, b):
        _check(lib.ora_per_token_cast(_ptr(x_bits[a:b]), b - a, C, group, f,
                                      _ptr(out[a:b]), _ptr(sf[a:b])), "per_token_cast")

    _row_parallel(T, threads, body)
    return out, sf


def cast_rows_f32(y: np.ndarray, fmt="e4m3", group: int = 128):
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, C = y.shape
    out = np.empty((T, C), np.uint8)
    sf = np.empty((T, C // group), np.float32)
    _check(lib.ora_cast_rows_f32(_ptr(y), T, C, group, _fmt(fmt), _ptr(out), _ptr(sf)),
           "cast_rows_f32")
    return out, sf


def cast_cols_f32(y: np.ndarray, fmt="e4m3", group: int = 128):
    """fp32 [T, C] -> (codes [C, T], sf_t [C, T/group]) with groups along tokens."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, C = y.shape
    out_t = np.empty((C, T), np.uint8)
    sf_t = np.empty((C, T // group), np.float32)
    _check(lib.ora_cast_cols_f32(_ptr(y), T, C, group, _fmt(fmt), _ptr(out_t), _ptr(sf_t)),
           "cast_cols_f32")
    return out_t, sf_t


class _Clamp:
    """The clamp arguments of the oracle's SwiGLU calls: a pointer to the fp32
    clamp value (None = no clamp) and a per-call counter of clamped values."""

    def __init__(self, clamp):
        self.on = clamp is not None
        self.value = ctypes.c_float(0.0 if clamp is None else float(clamp))
        self.lock = threading.Lock()
        self.total = 0

    def ptr(self):
        return ctypes.byref(self.value) if self.on else None

    def counter(self):
        return ctypes.c_int64(0)

    def add(self, c):
        with self.lock:
            self.total += int(c.value)


def swiglu_values(x_bits: np.ndarray, w: np.ndarray | None = None, threads: int = 1,
                  clamp: float | None = None):
    """x_bits: uint16 [T, 2H] (gate | up) -> fp32 y [T, H]; with ``clamp``,
    (y, number of clamped input values)."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H2 = x_bits.shape
    H = H2 // 2
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    y = np.empty((T, H), np.float32)
    cl = _Clamp(clamp)

    def body(a, b):
        n = cl.counter()
        _check(lib.ora_swiglu_values_clamp(_ptr(x_bits[a:b]), None if w is None else _ptr(w[a:b]),
                                           b - a, H, cl.ptr(), _ptr(y[a:b]), ctypes.byref(n)),
               "swiglu_values")
        cl.add(n)

    _row_parallel(T, threads, body)
    return (y, cl.total) if cl.on else y


def swiglu_cast(x_bits: np.ndarray, w: np.ndarray | None = None, fmt="e4m3",
                group: int = 128, threads: int = 1, clamp: float | None = None):
    """-> (codes [T, H], sf [T, H/group]); with ``clamp``, also the number of
    clamped input values."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H2 = x_bits.shape
    H = H2 // 2
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty((T, H), np.uint8)
    sf = np.empty((T, H // group), np.float32)
    f = _fmt(fmt)
    cl = _Clamp(clamp)

    def body(a, b):
        n = cl.counter()
        _check(lib.ora_swiglu_cast_clamp(_ptr(x_bits[a:b]), None if w is None else _ptr(w[a:b]),
                                         b - a, H, group, f, cl.ptr(), _ptr(out[a:b]),
                                         _ptr(sf[a:b]), ctypes.byref(n)), "swiglu_cast")
        cl.add(n)

    _row_parallel(T, threads, body)
    return (out, sf, cl.total) if cl.on else (out, sf)


def swiglu_cast_t(x_bits: np.ndarray, w: np.ndarray | None = None, fmt="e4m3",
                  group: int = 128, threads: int = 1, clamp: float | None = None):
    """-> (codes [T, H], sf [T, H/group], codes_t [H, T], sf_t [H, T/group]);
    with ``clamp``, also the number of clamped input values."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H2 = x_bits.shape
    H = H2 // 2
    if T % group:
        raise ValueError("T must be a multiple of group")
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty((T, H), np.uint8)
    sf = np.empty((T, H // group), np.float32)
    out_t = np.empty((H, T), np.uint8)
    sf_t = np.empty((H, T // group), np.float32)
    f = _fmt(fmt)
    cl = _Clamp(clamp)

    # Row blocks of `group` tokens are independent: run each block as its own
    # oracle problem and scatter its column outputs into the [H, T] arrays.
    def body(a, b):
        n = b - a
        o_t = np.empty((H, n), np.uint8)
        s_t = np.empty((H, n // group), np.float32)
        cnt = cl.counter()
        _check(lib.ora_swiglu_cast_t_clamp(_ptr(x_bits[a:b]), None if w is None else _ptr(w[a:b]),
                                           n, H, group, f, cl.ptr(), _ptr(out[a:b]),
                                           _ptr(sf[a:b]), _ptr(o_t), _ptr(s_t),
                                           ctypes.byref(cnt)), "swiglu_cast_t")
        cl.add(cnt)
        out_t[:, a:b] = o_t
        sf_t[:, a // group:b // group] = s_t

    _row_parallel(T, threads, body, align=group)
    res = (out, sf, out_t, sf_t)
    return res + (cl.total,) if cl.on else res


def swiglu_backward_values(x_bits: np.ndarray, dy_bits: np.ndarray, w: np.ndarray | None = None,
                           threads: int = 1):
    """x_bits: uint16 [T, 2H] (gate | up), dy_bits: uint16 [T, H] -> fp32 [T, 2H] = [dg | du]."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    dy_bits = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    T, H2 = x_bits.shape
    H = H2 // 2
    assert dy_bits.shape == (T, H)
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    grad = np.empty((T, 2 * H), np.float32)

    def body(a, b):
        _check(lib.ora_swiglu_backward_values(_ptr(x_bits[a:b]), _ptr(dy_bits[a:b]),
                                              None if w is None else _ptr(w[a:b]), b - a, H,
                                              _ptr(grad[a:b])), "swiglu_backward_values")

    _row_parallel(T, threads, body)
    return grad


def swiglu_backward_cast(x_bits: np.ndarray, dy_bits: np.ndarray, w: np.ndarray | None = None,
                         fmt="e4m3", group: int = 128, threads: int = 1):
    """-> (codes [T, 2H] of [dg | du], sf [T, 2H/group])."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    dy_bits = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    T, H2 = x_bits.shape
    H = H2 // 2
    assert dy_bits.shape == (T, H)
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty((T, 2 * H), np.uint8)
    sf = np.empty((T, 2 * H // group), np.float32)
    f = _fmt(fmt)

    def body(a, b):
        _check(lib.ora_swiglu_backward_cast(_ptr(x_bits[a:b]), _ptr(dy_bits[a:b]),
                                            None if w is None else _ptr(w[a:b]), b - a, H, group,
                                            f, _ptr(out[a:b]), _ptr(sf[a:b])),
               "swiglu_backward_cast")

    _row_parallel(T, threads, body)
    return out, sf


# --------------------------------------------------------------------------
# scale-factor layout options
# --------------------------------------------------------------------------

SF_ROUND_POW2 = 1
SF_UE8M0_PACKED = 2
SF_COL_MAJOR = 4
# codes of fl32(v * fl32(1 / s)) instead of fl32(v / s); scales unchanged
Q_RECIPROCAL = 8


def pow2_ceil(s: float) -> np.float32:
    return np.float32(_load().ora_pow2_ceil(float(np.float32(s))))


def sf_shape(T: int, G: int, flags: int):
    """(shape, dtype) of the scale output for T rows of G groups."""
    T4 = (T + 3) // 4 * 4
    W = (G + 3) // 4
    if flags & SF_UE8M0_PACKED:
        return ((W, T4) if flags & SF_COL_MAJOR else (T, W)), np.uint32
    return ((G, T4) if flags & SF_COL_MAJOR else (T, G)), np.float32


def cast_rows_f32_ex(y: np.ndarray, fmt="e4m3", group: int = 128, flags: int = 0,
                     threads: int = 1):
    """fp32 [T, C] -> (codes [T, C], scales in the layout `flags` selects).
    Row blocks of 4 rows are independent, so ``threads`` splits 4-aligned row
    ranges (column-major layouts are gathered after)."""
    lib = _load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    T, C = y.shape
    if group <= 0 or C % group:
        raise ValueError("group must divide C")
    G = C // group
    out = np.empty((T, C), np.uint8)
    shape, dt = sf_shape(T, G, flags)
    sf = np.empty(shape, dt)
    f = _fmt(fmt)
    if threads <= 1 or T < 8:
        _check(lib.ora_cast_rows_f32_ex(_ptr(y), T, C, group, f, flags, _ptr(out), _ptr(sf)),
               "cast_rows_f32_ex")
        return out, sf

    def body(a, b):
        part_shape, _ = sf_shape(b - a, G, flags)
        part = np.empty(part_shape, dt)
        _check(lib.ora_cast_rows_f32_ex(_ptr(y[a:b]), b - a, C, group, f, flags,
                                        _ptr(out[a:b]), _ptr(part)), "cast_rows_f32_ex")
        if flags & SF_COL_MAJOR:
            n = part.shape[1]
            sf[:, a:a + n] = part
        else:
            sf[a:b] = part

    _row_parallel(T, threads, body, align=4)
    return out, sf


def per_token_cast_ex(x_bits: np.ndarray, fmt="e4m3", group: int = 128, flags: int = 0,
                      threads: int = 1):
    """bf16 [T, C] (exact widening to fp32) -> the cast with scale options."""
    xf = (np.ascontiguousarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return cast_rows_f32_ex(xf, fmt, group, flags, threads)


# --------------------------------------------------------------------------
# per-channel / per-block casts and cast back
# --------------------------------------------------------------------------

def per_channel_cast(x_bits: np.ndarray, fmt="e4m3", group: int = 128, transpose: bool = False,
                     threads: int = 1):
    """bf16 [T, C] -> codes ([T, C], or [C, T] with transpose) and scales
    ([T/group, C], or [C, T/group]) with groups of `group` tokens per channel."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, C = x_bits.shape
    if group <= 0 or T % group:
        raise ValueError("T must be a multiple of group")
    f = _fmt(fmt)
    out = np.empty((C, T) if transpose else (T, C), np.uint8)
    sf = np.empty((C, T // group) if transpose else (T // group, C), np.float32)
    if threads <= 1 or C < 256:
        _check(lib.ora_per_channel_cast(_ptr(x_bits), T, C, group, f, int(transpose),
                                        _ptr(out), _ptr(sf)), "per_channel_cast")
        return out, sf

    # independent row blocks of `group` tokens
    def body(a, b):
        n = b - a
        o = np.empty((C, n) if transpose else (n, C), np.uint8)
        s = np.empty((C, n // group) if transpose else (n // group, C), np.float32)
        _check(lib.ora_per_channel_cast(_ptr(np.ascontiguousarray(x_bits[a:b])), n, C, group, f,
                                        int(transpose), _ptr(o), _ptr(s)), "per_channel_cast")
        if transpose:
            out[:, a:b] = o
            sf[:, a // group:b // group] = s
        else:
            out[a:b] = o
            sf[a // group:b // group] = s

    _row_parallel(T, threads, body, align=group)
    return out, sf


def per_block_cast(x_bits: np.ndarray, fmt="e4m3", block: int = 128, threads: int = 1):
    """bf16 [T, C] -> (codes [T, C], scales [ceil(T/block), C/block])."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, C = x_bits.shape
    if block <= 0 or C % block:
        raise ValueError("block must divide C")
    f = _fmt(fmt)
    out = np.empty((T, C), np.uint8)
    sf = np.empty((-(-T // block), C // block), np.float32)

    def body(a, b):
        _check(lib.ora_per_block_cast(_ptr(x_bits[a:b]), b - a, C, block, f, _ptr(out[a:b]),
                                      _ptr(sf[a // block:-(-b // block)])), "per_block_cast")

    _row_parallel(T, threads, body, align=block)
    return out, sf


def cast_back(codes: np.ndarray, sf: np.ndarray, group_rows: int = 1, group_cols: int = 128,
              fmt="e4m3", threads: int = 1) -> np.ndarray:
    """codes uint8 [T, C], sf fp32 [ceil(T/gr), C/gc] -> fp32 [T, C] = decode * scale."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.float32)
    T, C = codes.shape
    out = np.empty((T, C), np.float32)
    f = _fmt(fmt)

    def body(a, b):
        _check(lib.ora_cast_back(_ptr(codes[a:b]), _ptr(sf[a // group_rows:]), b - a, C,
                                 group_rows, group_cols, f, _ptr(out[a:b])), "cast_back")

    _row_parallel(T, threads, body, align=group_rows)
    return out
