"""Seeded synthetic inputs for the quantization workloads.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle: it only draws random numbers and rounds them to bf16 bit patterns.
It holds none of the quantization arithmetic (no scales, no FP8 codes, no
SwiGLU).  Every array it returns is host memory (numpy).

Rows are generated in fixed chunks of ``CHUNK_ROWS`` rows, each chunk from its
own PCG64 stream keyed by (seed, workload, chunk index).  The result does not
depend on how many threads generate it, and a workload cut to fewer rows is a
prefix of the full-size workload.

Workloads (all seeded, no dataset involved):

* ``plain_small``   bf16 [1024, 4096], N(0, 1).
* ``plain_outlier`` bf16 [8192, 7168], N(0, 1); 0.1% of the entries, chosen by
  the generator, multiplied by 100; rows 0, 1024, 2048, ... all zero.
* ``swiglu``        bf16 [16384, 4096] = gate | up with gate ~ N(0, 2) (standard
  deviation 2) and up ~ N(0, 1); H = 2048.
* ``swiglu_moe``    bf16 [65536, 4096] N(0, 1) (8192 tokens x top-8 rows) and
  a fp32 routing weight per row: Uniform(0.01, 1) normalised over the 8 rows of
  each token.
* ``swiglu_t``      bf16 [131072, 4096] N(0, 1), for the cast + transposed cast.
* ``swiglu_bwd``    bf16 [65536, 4096] N(0, 1) gate|up, an upstream gradient dy
  bf16 [65536, 2048] N(0, 1) and the routing weights of ``swiglu_moe``.
* ``per_channel``   bf16 [16384, 7168] N(0, 1) with every 64th channel (from
  channel 0) multiplied by 20: a few outlier channels, the case a per-channel
  scale serves.
* ``per_block``     bf16 [16320, 7168] drawn like ``plain_outlier`` (without the
  zero rows); 16320 tokens leave a last block row of 64 tokens.
* ``cast_back``     uint8 [16384, 7168] codes, uniform over all 256 byte values,
  and fp32 per-token scales [16384, 56] log-uniform in [2^-22, 2^4].
* ``plain_f32``     fp32 [8192, 7168] drawn like ``plain_outlier`` but kept in
  binary32 (an fp32 activation, e.g. a gradient before its cast).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK_ROWS = 1024

WORKLOADS = {
    # name: (rows, cols, description)
    "plain_small": (1024, 4096, "per_token_cast E4M3, x bf16 [1024, 4096] ~ N(0,1)"),
    "plain_outlier": (8192, 7168, "per_token_cast E4M3/E5M2, x bf16 [8192, 7168] ~ N(0,1), "
                                  "0.1% outliers x100, one all-zero row per 1024"),
    "swiglu": (16384, 4096, "swiglu + per-token E4M3 cast, bf16 [16384, 4096] "
                            "gate~N(0,2) | up~N(0,1), H=2048"),
    "swiglu_moe": (65536, 4096, "swiglu x routing weight + per-token E4M3 cast, "
                                "bf16 [65536, 4096] ~ N(0,1), 8192 tokens x top-8, H=2048"),
    "swiglu_t": (131072, 4096, "swiglu + per-token E4M3 cast + transposed cast, "
                               "bf16 [131072, 4096] ~ N(0,1), H=2048"),
    "swiglu_bwd": (65536, 4096, "swiglu backward x routing weight + per-token E4M3 cast of "
                                "[dgate | dup], bf16 [65536, 4096] ~ N(0,1) and dy bf16 "
                                "[65536, 2048] ~ N(0,1), 8192 tokens x top-8, H=2048"),
    "per_channel": (16384, 7168, "per_channel_cast (+transpose) E4M3, x bf16 [16384, 7168] "
                                 "~ N(0,1), every 64th channel x20"),
    "per_block": (16320, 7168, "per_block_cast E4M3, x bf16 [16320, 7168] ~ N(0,1), 0.1% "
                               "outliers x100, last block row 64 tokens"),
    "cast_back": (16384, 7168, "cast_back E4M3 -> bf16 with per-token scales, codes uint8 "
                               "[16384, 7168] uniform bytes, scales fp32 [16384, 56] "
                               "log-uniform in [2^-22, 2^4]"),
    "plain_f32": (8192, 7168, "per_token_cast E4M3 of an fp32 input, x fp32 [8192, 7168] "
                              "~ N(0,1), 0.1% outliers x100, one all-zero row per 1024"),
}

_WORKLOAD_IDS = {name: i + 1 for i, name in enumerate(WORKLOADS)}


def rng_for(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest, ties to even); return uint16 bits.
    Inputs must be finite.  Works on a copy."""
    u = np.array(v, dtype=np.float32, order="C", copy=True).view(np.uint32)
    _round_inplace(u)
    return np.ascontiguousarray(u.view(np.uint16)[..., 1::2]) if u.ndim else \
        np.uint16(int(u) >> 16)


def _round_inplace(u: np.ndarray) -> None:
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    u += np.uint32(0x7FFF)
    u += lsb


def _to_bf16_into(v: np.ndarray, dst: np.ndarray) -> None:
    """Round float32 ``v`` (modified in place) to bf16 bits written into ``dst``."""
    u = v.view(np.uint32)
    _round_inplace(u)
    dst[...] = u.view(np.uint16)[..., 1::2]


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _chunked(T: int, fill, row_begin: int = 0) -> None:
    """Run fill(chunk_index, lo, hi, dst) over the fixed row chunks that cover
    rows [row_begin, row_begin + T) of the stream: chunk i keeps its local rows
    [lo, hi) and writes them to the output rows ``dst`` (a slice).  Each fill
    draws a whole chunk's worth of numbers, so any row range holds the same
    values as the same rows of a longer draw."""
    T, row_begin = int(T), int(row_begin)
    if T <= 0:
        return
    first, last = row_begin // CHUNK_ROWS, (row_begin + T - 1) // CHUNK_ROWS

    def one(i):
        a = max(row_begin, i * CHUNK_ROWS)
        b = min(row_begin + T, (i + 1) * CHUNK_ROWS)
        fill(i, a - i * CHUNK_ROWS, b - i * CHUNK_ROWS, slice(a - row_begin, b - row_begin))

    if first == last:
        one(first)
        return
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(first, last + 1)))


def normal_bf16(seed: int, stream: int, T: int, C: int, std: float = 1.0,
                row_begin: int = 0) -> np.ndarray:
    """bf16 bits of a [T, C] matrix of N(0, std^2) samples (rows row_begin ..
    row_begin + T - 1 of the stream)."""
    out = np.empty((int(T), int(C)), np.uint16)

    def fill(i, a, b, dst):
        v = rng_for(seed, stream, i).standard_normal((CHUNK_ROWS, C), dtype=np.float32)[a:b]
        if std != 1.0:
            v *= np.float32(std)
        _to_bf16_into(v, out[dst])

    _chunked(T, fill, row_begin)
    return out


def outlier_bf16(seed: int, stream: int, T: int, C: int, frac: float = 1e-3,
                 factor: float = 100.0, zero_row_every: int = 1024,
                 as_f32: bool = False, row_begin: int = 0) -> np.ndarray:
    """N(0,1) with a fraction ``frac`` of entries, chosen by the generator,
    multiplied by ``factor`` and every ``zero_row_every``-th row of the stream
    (from row 0) zero.  bf16 bits, or the binary32 values themselves with
    ``as_f32``; rows row_begin .. row_begin + T - 1 of the stream."""
    out = np.empty((int(T), int(C)), np.float32 if as_f32 else np.uint16)

    def fill(i, a, b, dst):
        rng = rng_for(seed, stream, i)
        v = rng.standard_normal((CHUNK_ROWS, C), dtype=np.float32)[a:b]
        mask = rng.random((CHUNK_ROWS, C), dtype=np.float32)[a:b] < np.float32(frac)
        v[mask] *= np.float32(factor)
        if as_f32:
            out[dst] = v
        else:
            _to_bf16_into(v, out[dst])

    _chunked(T, fill, row_begin)
    if zero_row_every:
        out[(-int(row_begin)) % zero_row_every::zero_row_every] = 0
    return out


def swiglu_bf16(seed: int, stream: int, T: int, H: int, gate_std: float = 1.0,
                up_std: float = 1.0, row_begin: int = 0) -> np.ndarray:
    """bf16 bits of a [T, 2H] gate | up matrix (rows row_begin .. row_begin + T - 1
    of the stream)."""
    out = np.empty((int(T), 2 * int(H)), np.uint16)

    def fill(i, a, b, dst):
        rng = rng_for(seed, stream, i)
        g = rng.standard_normal((CHUNK_ROWS, H), dtype=np.float32)[a:b]
        if gate_std != 1.0:
            g *= np.float32(gate_std)
        u = rng.standard_normal((CHUNK_ROWS, H), dtype=np.float32)[a:b]
        if up_std != 1.0:
            u *= np.float32(up_std)
        _to_bf16_into(g, out[dst, :H])
        _to_bf16_into(u, out[dst, H:])

    _chunked(T, fill, row_begin)
    return out


def channel_outlier_bf16(seed: int, stream: int, T: int, C: int, every: int = 64,
                         factor: float = 20.0, row_begin: int = 0) -> np.ndarray:
    """N(0,1) with every ``every``-th channel (from channel 0) multiplied by
    ``factor`` (rows row_begin .. row_begin + T - 1 of the stream)."""
    out = np.empty((int(T), int(C)), np.uint16)

    def fill(i, a, b, dst):
        v = rng_for(seed, stream, i).standard_normal((CHUNK_ROWS, C), dtype=np.float32)[a:b]
        v[:, ::every] *= np.float32(factor)
        _to_bf16_into(v, out[dst])

    _chunked(T, fill, row_begin)
    return out


def random_bytes(seed: int, stream: int, T: int, C: int, row_begin: int = 0) -> np.ndarray:
    """uint8 [T, C], every byte value equally likely (rows row_begin ..
    row_begin + T - 1 of the stream)."""
    out = np.empty((int(T), int(C)), np.uint8)

    def fill(i, a, b, dst):
        out[dst] = rng_for(seed, stream, i).integers(0, 256, (CHUNK_ROWS, C), np.uint8)[a:b]

    _chunked(T, fill, row_begin)
    return out


def log_uniform_f32(seed: int, stream: int, shape, lo_exp: float, hi_exp: float) -> np.ndarray:
    """fp32 values 2^u with u ~ Uniform(lo_exp, hi_exp)."""
    u = rng_for(seed, stream, 1 << 21).uniform(lo_exp, hi_exp, size=shape)
    return np.ascontiguousarray(np.exp2(u).astype(np.float32))


def routing_weights(seed: int, stream: int, tokens: int, topk: int = 8) -> np.ndarray:
    """fp32 [tokens * topk]: Uniform(0.01, 1) normalised over each token's rows."""
    raw = rng_for(seed, stream, 1 << 20).uniform(0.01, 1.0, size=(int(tokens), int(topk)))
    w = raw / raw.sum(axis=1, keepdims=True)
    return np.ascontiguousarray(w.astype(np.float32).reshape(-1))


def workload(name: str, seed: int = 0, rows: int | None = None, row_begin: int = 0) -> dict:
    """Inputs of a named workload: dict with ``x`` (uint16 bf16 bits, row-major)
    and, for the weighted SwiGLU, ``w`` (fp32, one per row).  ``rows`` cuts the
    workload to its first rows (same distribution), which quick tests use.
    ``row_begin`` shifts the window: the result is rows [row_begin, row_begin +
    rows) of one longer draw of the same workload (a shard of a batch of several
    workloads' worth of rows, as the ranks of a multi-GPU run quantize it)."""
    if name not in WORKLOADS:
        raise KeyError(name)
    T, C, _ = WORKLOADS[name]
    if rows is not None:
        T = int(rows)
    a = int(row_begin)
    if a < 0:
        raise ValueError("row_begin must be >= 0")
    sid = _WORKLOAD_IDS[name]
    if name == "plain_small":
        return {"x": normal_bf16(seed, sid, T, C, row_begin=a)}
    if name == "plain_outlier":
        return {"x": outlier_bf16(seed, sid, T, C, row_begin=a)}
    if name == "swiglu":
        return {"x": swiglu_bf16(seed, sid, T, C // 2, gate_std=2.0, up_std=1.0, row_begin=a)}
    if name in ("swiglu_moe", "swiglu_bwd"):
        topk = 8
        # the weights of every token up to the window's end, then the window
        w = routing_weights(seed, sid, -(-(a + T) // topk), topk)[a:a + T]
        d = {"x": swiglu_bf16(seed, sid, T, C // 2, row_begin=a)}
        if name == "swiglu_bwd":
            d["dy"] = normal_bf16(seed, sid + 100, T, C // 2, row_begin=a)
        d["w"] = np.ascontiguousarray(w)
        return d
    if name == "swiglu_t":
        return {"x": swiglu_bf16(seed, sid, T, C // 2, row_begin=a)}
    if name == "per_channel":
        return {"x": channel_outlier_bf16(seed, sid, T, C, row_begin=a)}
    if name == "per_block":
        return {"x": outlier_bf16(seed, sid, T, C, zero_row_every=0, row_begin=a)}
    if name == "plain_f32":
        return {"x": outlier_bf16(seed, sid, T, C, as_f32=True, row_begin=a)}
    if name == "cast_back":
        sf = log_uniform_f32(seed, sid, (a + T, C // 128), -22.0, 4.0)[a:]
        return {"codes": random_bytes(seed, sid, T, C, row_begin=a),
                "sf": np.ascontiguousarray(sf)}
    raise KeyError(name)
