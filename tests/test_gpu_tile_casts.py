"""Parity of the per-channel cast, the per-block cast and cast back (through the
C ABI) with the CPU oracle.  All three are bit-exact: codes and scales of the
casts byte for byte, cast-back outputs bit for bit (NaN codes give NaN on both
sides).  Every output buffer is surrounded by guard bytes that must stay
untouched.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests import parity
from tests.test_gpu_parity import Guarded, stream_of, to_dev_bf16

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def run_channel(x_bits, fmt, dev, transpose):
    T, C = x_bits.shape
    xd = to_dev_bf16(x_bits, dev)
    out = Guarded(T * C, dev)
    sf = Guarded((T // 128) * C * 4, dev)
    st = tkq.tkq_per_channel_cast(ctypes.c_void_p(xd.data_ptr()), out.ptr, sf.ptr, T, C, 128,
                                  oracle.FMT[fmt], int(transpose), stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    if transpose:
        return out.data().reshape(C, T), sf.data().view(np.float32).reshape(C, T // 128)
    return out.data().reshape(T, C), sf.data().view(np.float32).reshape(T // 128, C)


def run_block(x_bits, fmt, dev):
    T, C = x_bits.shape
    nb = -(-T // 128)
    xd = to_dev_bf16(x_bits, dev)
    out = Guarded(T * C, dev)
    sf = Guarded(nb * (C // 128) * 4, dev)
    st = tkq.tkq_per_block_cast(ctypes.c_void_p(xd.data_ptr()), out.ptr, sf.ptr, T, C, 128,
                                oracle.FMT[fmt], stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    return out.data().reshape(T, C), sf.data().view(np.float32).reshape(nb, C // 128)


def run_cast_back(codes, sf, gr, gc, fmt, bf16, dev):
    T, C = codes.shape
    cd = torch.from_numpy(np.ascontiguousarray(codes)).to(dev)
    sd = torch.from_numpy(np.ascontiguousarray(sf, np.float32)).to(dev)
    out = Guarded(T * C * (2 if bf16 else 4), dev)
    st = tkq.tkq_cast_back(ctypes.c_void_p(cd.data_ptr()), ctypes.c_void_p(sd.data_ptr()),
                           out.ptr, T, C, gr, gc, oracle.FMT[fmt],
                           tkq.OUT_BF16 if bf16 else tkq.OUT_F32, stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    return out.data().view(np.uint16 if bf16 else np.uint32).reshape(T, C)


def expected_cast_back(codes, sf, gr, gc, fmt, bf16):
    """The oracle's fp32 result; for bf16 output rounded to nearest even by
    PyTorch's CPU conversion.  Returned as raw bits."""
    y = oracle.cast_back(codes, sf, gr, gc, fmt, threads=THREADS)
    if bf16:
        return torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return y.view(np.uint32)


def assert_bits_equal_nan_aware(name, got, exp, bf16):
    nan_mask = (0x7F80, 0x007F) if bf16 else (0x7F800000, 0x007FFFFF)
    e_nan = ((exp & nan_mask[0]) == nan_mask[0]) & ((exp & nan_mask[1]) != 0)
    g_nan = ((got & nan_mask[0]) == nan_mask[0]) & ((got & nan_mask[1]) != 0)
    assert np.array_equal(e_nan, g_nan), f"{name}: NaN positions differ"
    parity.assert_bit_exact(name, np.where(e_nan, 0, got).astype(got.dtype),
                            np.where(e_nan, 0, exp).astype(exp.dtype))


# ---------------------------------------------------------------------------
# per-channel cast
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("transpose", [False, True])
def test_per_channel_full_workload(cuda_device, transpose):
    x = synth.workload("per_channel")["x"]
    codes, sf = run_channel(x, "e4m3", cuda_device, transpose)
    e_codes, e_sf = oracle.per_channel_cast(x, "e4m3", transpose=transpose, threads=THREADS)
    parity.assert_bit_exact("sf", sf, e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)


@pytest.mark.parametrize("T", [128, 256, 1152])
@pytest.mark.parametrize("C", [128, 384, 2048])
@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_per_channel_shapes(cuda_device, T, C, transpose, fmt):
    x = synth.outlier_bf16(11, T + C, T, C, zero_row_every=0)
    x[:, 5] = 0                      # an all-zero channel: the 1e-4 floor
    x[:, 6] = 0x8000                 # an all -0 channel: signed zeros kept
    codes, sf = run_channel(x, fmt, cuda_device, transpose)
    e_codes, e_sf = oracle.per_channel_cast(x, fmt, transpose=transpose)
    parity.assert_bit_exact("sf", sf, e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)


def test_per_channel_is_per_token_of_the_transpose_on_gpu(cuda_device):
    """The transposed per-channel output equals the per-token cast of x^T, both
    computed on the GPU (a layout check independent of the oracle)."""
    T, C = 512, 256
    x = synth.normal_bf16(3, 4, T, C)
    xd = to_dev_bf16(x, cuda_device)
    ct, st = tkq.per_channel_cast(xd, transpose=True)
    cp, sp = tkq.per_token_cast(xd.t().contiguous())
    assert torch.equal(ct.view(torch.uint8), cp.view(torch.uint8))
    assert torch.equal(st, sp)


# ---------------------------------------------------------------------------
# per-block cast
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_per_block_full_workload(cuda_device, fmt):
    x = synth.workload("per_block")["x"]
    codes, sf = run_block(x, fmt, cuda_device)
    e_codes, e_sf = oracle.per_block_cast(x, fmt, threads=THREADS)
    parity.assert_bit_exact("sf", sf, e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)


@pytest.mark.parametrize("T", [1, 7, 128, 129, 1031])
@pytest.mark.parametrize("C", [128, 384, 7168])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_per_block_ragged(cuda_device, T, C, fmt):
    x = synth.outlier_bf16(12, T + C, T, C, zero_row_every=0)
    if C >= 384:
        x[:, 128:256] = 0            # one all-zero block column
    codes, sf = run_block(x, fmt, cuda_device)
    e_codes, e_sf = oracle.per_block_cast(x, fmt)
    parity.assert_bit_exact("sf", sf, e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)


def test_per_block_tiny_last_block_not_diluted(cuda_device):
    """A short last block row takes its amax from its own rows only: a large
    value in block row 0 must not leak into the 1-row block row 1."""
    T, C = 129, 128
    x = synth.normal_bf16(5, 6, T, C)
    x[0, 0] = synth.f32_to_bf16_bits(np.float32(1000.0))
    codes, sf = run_block(x, "e4m3", cuda_device)
    e_codes, e_sf = oracle.per_block_cast(x, "e4m3")
    parity.assert_bit_exact("sf", sf, e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)
    assert sf[1, 0] < sf[0, 0] / 50


# ---------------------------------------------------------------------------
# cast back
# ---------------------------------------------------------------------------

GRANULARITIES = [(1, 128), (128, 1), (128, 128)]


@pytest.mark.parametrize("gr,gc", GRANULARITIES)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("T,C", [(1, 128), (300, 384), (1031, 2048)])
def test_cast_back_every_code(cuda_device, gr, gc, fmt, bf16, T, C):
    codes = synth.random_bytes(21, T * 7 + C, T, C)
    codes[0, :128] = np.arange(128, dtype=np.uint8)     # every code appears
    if T > 1:
        codes[1, :128] = np.arange(128, 256).astype(np.uint8)
    sf = synth.log_uniform_f32(22, T + C, (-(-T // gr), C // gc), -22.0, 4.0)
    got = run_cast_back(codes, sf, gr, gc, fmt, bf16, cuda_device)
    exp = expected_cast_back(codes, sf, gr, gc, fmt, bf16)
    assert_bits_equal_nan_aware("cast_back", got, exp, bf16)


@pytest.mark.parametrize("bf16", [False, True])
def test_cast_back_full_workload(cuda_device, bf16):
    w = synth.workload("cast_back")
    got = run_cast_back(w["codes"], w["sf"], 1, 128, "e4m3", bf16, cuda_device)
    exp = expected_cast_back(w["codes"], w["sf"], 1, 128, "e4m3", bf16)
    assert_bits_equal_nan_aware("cast_back", got, exp, bf16)


def test_cast_back_subnormal_products(cuda_device):
    """Scales that push products below 2^-126 must give binary32 subnormals
    (no flush to zero)."""
    T, C = 4, 128
    codes = synth.random_bytes(31, 32, T, C)
    sf = np.full((T, 1), 2.0 ** -130, np.float32)
    got = run_cast_back(codes, sf, 1, 128, "e4m3", False, cuda_device)
    exp = expected_cast_back(codes, sf, 1, 128, "e4m3", False)
    assert_bits_equal_nan_aware("cast_back", got, exp, False)
    assert np.any((got & 0x7F800000) == 0) and np.any(got & 0x007FFFFF)


@pytest.mark.parametrize("kind", ["token", "channel", "block"])
def test_round_trip_through_gpu_casts(cuda_device, kind):
    """Cast then cast back on the GPU equals the oracle's cast then cast back."""
    T, C = 1024, 512
    x = synth.outlier_bf16(41, 42, T, C, zero_row_every=0)
    xd = to_dev_bf16(x, cuda_device)
    if kind == "token":
        q, s = tkq.per_token_cast(xd)
        gs, (eq, es) = (1, 128), oracle.per_token_cast(x, "e4m3")
    elif kind == "channel":
        q, s = tkq.per_channel_cast(xd)
        gs, (eq, es) = (128, 1), oracle.per_channel_cast(x, "e4m3")
    else:
        q, s = tkq.per_block_cast(xd)
        gs, (eq, es) = (128, 128), oracle.per_block_cast(x, "e4m3")
    y = tkq.cast_back(q, s, group_size=gs)
    ey = oracle.cast_back(eq, es, gs[0], gs[1], "e4m3")
    parity.assert_bit_exact("round trip", y.cpu().numpy(), ey)


def test_tensor_api_shapes_and_dtypes(cuda_device):
    x = to_dev_bf16(synth.normal_bf16(1, 2, 384, 256), cuda_device)
    q, s = tkq.per_channel_cast(x, fmt="e5m2")
    assert q.shape == (384, 256) and q.dtype == torch.float8_e5m2 and s.shape == (3, 256)
    q, s = tkq.per_channel_cast(x, transpose=True)
    assert q.shape == (256, 384) and q.dtype == torch.float8_e4m3fn and s.shape == (256, 3)
    q, s = tkq.per_block_cast(x[:300])
    assert q.shape == (300, 256) and s.shape == (3, 2)
    y = tkq.cast_back(q, s, group_size=(128, 128), out_dtype=torch.bfloat16)
    assert y.shape == (300, 256) and y.dtype == torch.bfloat16
    with pytest.raises(ValueError):
        tkq.cast_back(q, s, group_size=(1, 128))
    with pytest.raises(tkq.TkqError):
        tkq.per_channel_cast(x[:300])                    # T % 128


@pytest.mark.slow
def test_beyond_2_31_elements(cuda_device):
    """x of 131,200 x 16,384 bf16 (2.15e9 elements, 4.3 GB): byte offsets beyond
    2^32 in every kernel.  The per-channel cast (transposed and in place), the
    per-block cast (with a short last block row) and cast back of the per-block
    result are checked bit-exact on sampled 128-token blocks at both ends and in
    the middle."""
    T, C = 131_200, 16_384
    dev = cuda_device
    rng = np.random.default_rng(78)
    nb = T // 128
    blocks = sorted({0, 1, nb // 2, nb - 2, nb - 1})
    keep = {}
    xd = torch.empty((T, C), dtype=torch.int16, device=dev)
    chunk = 16384
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        bits = rng.integers(0, 1 << 16, size=(b - a, C), dtype=np.uint16)
        e = rng.integers(127 - 20, 127 + 12, size=(b - a, C), dtype=np.uint16)
        bits = (bits & np.uint16(0x807F)) | (e << np.uint16(7)).astype(np.uint16)
        xd[a:b] = torch.from_numpy(bits.view(np.int16)).to(dev)
        for k in blocks:
            if a <= 128 * k < b:
                keep[k] = bits[128 * k - a:128 * k - a + 128].copy()
    xb = xd.view(torch.bfloat16)
    st = stream_of(dev)

    # per-channel, transposed: out_t [C, T], sf_t [C, T/128]
    out = torch.empty((C, T), dtype=torch.uint8, device=dev)
    sf = torch.empty((C, nb), dtype=torch.float32, device=dev)
    assert tkq.tkq_per_channel_cast(ctypes.c_void_p(xb.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(sf.data_ptr()), T, C, 128, 0, 1, st) == 0
    torch.cuda.synchronize()
    for k in blocks:
        ro, rs = oracle.per_channel_cast(keep[k], "e4m3", transpose=True, threads=THREADS)
        parity.assert_bit_exact(f"transposed codes, block {k}",
                                out[:, 128 * k:128 * k + 128].cpu().numpy(), ro)
        parity.assert_bit_exact(f"transposed scales, block {k}", sf[:, k:k + 1].cpu().numpy(), rs)
    del out, sf

    # per-channel, in place: out [T, C], sf [T/128, C]
    out = torch.empty((T, C), dtype=torch.uint8, device=dev)
    sf = torch.empty((nb, C), dtype=torch.float32, device=dev)
    assert tkq.tkq_per_channel_cast(ctypes.c_void_p(xb.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(sf.data_ptr()), T, C, 128, 0, 0, st) == 0
    torch.cuda.synchronize()
    for k in blocks:
        ro, rs = oracle.per_channel_cast(keep[k], "e4m3", threads=THREADS)
        parity.assert_bit_exact(f"in-place codes, block {k}",
                                out[128 * k:128 * k + 128].cpu().numpy(), ro)
        parity.assert_bit_exact(f"in-place scales, block {k}", sf[k:k + 1].cpu().numpy(), rs)
    del out, sf

    # per-block on the first T - 64 rows (the last block row holds 64 tokens)
    Tb = T - 64
    out = torch.empty((Tb, C), dtype=torch.uint8, device=dev)
    sf = torch.empty((nb, C // 128), dtype=torch.float32, device=dev)
    assert tkq.tkq_per_block_cast(ctypes.c_void_p(xb.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_void_p(sf.data_ptr()), Tb, C, 128, 0, st) == 0
    torch.cuda.synchronize()
    # cast back of the per-block result to bf16
    y = torch.empty((Tb, C), dtype=torch.bfloat16, device=dev)
    assert tkq.tkq_cast_back(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
                             ctypes.c_void_p(y.data_ptr()), Tb, C, 128, 128, 0, tkq.OUT_BF16,
                             st) == 0
    torch.cuda.synchronize()
    for k in blocks:
        rows = keep[k][:max(0, min(128, Tb - 128 * k))]
        ro, rs = oracle.per_block_cast(rows, "e4m3")
        got = out[128 * k:128 * k + rows.shape[0]].cpu().numpy()
        parity.assert_bit_exact(f"per-block codes, block {k}", got, ro)
        parity.assert_bit_exact(f"per-block scales, block {k}", sf[k:k + 1].cpu().numpy(), rs)
        ey = expected_cast_back(ro, rs, 128, 128, "e4m3", True)
        gy = y[128 * k:128 * k + rows.shape[0]].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_bits_equal_nan_aware(f"cast back, block {k}", gy, ey, True)


@pytest.mark.slow
def test_repeated_launches_are_identical_for_every_kernel(cuda_device):
    """60 launches of every other kernel on one input (full-size workloads):
    each result equals the first bit for bit, which equals the oracle for the
    exact casts.  A ring stage handed back to the TMA producer before its
    readers are done, or a missing barrier between a group's table writes and
    reads, shows up here as a rare differing group."""
    dev = cuda_device
    xc = synth.workload("per_channel")["x"]
    xb = synth.workload("per_block")["x"]
    xcd, xbd = to_dev_bf16(xc, dev), to_dev_bf16(xb, dev)
    moe = synth.workload("swiglu_moe")
    xs = to_dev_bf16(moe["x"], dev)
    ws = torch.from_numpy(moe["w"]).to(dev)
    bwd = synth.workload("swiglu_bwd", rows=16384)
    xg, dy = to_dev_bf16(bwd["x"], dev), to_dev_bf16(bwd["dy"], dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    ops = {
        "per_channel": lambda: tkq.per_channel_cast(xcd),
        "per_channel_t": lambda: tkq.per_channel_cast(xcd, transpose=True),
        "per_block": lambda: tkq.per_block_cast(xbd),
        "swiglu": lambda: tkq.swiglu_forward_and_per_token_cast(xs, topk_weights=ws),
        "swiglu_clamp": lambda: tkq.swiglu_forward_and_per_token_cast(
            xs, use_clamp=True, swiglu_clamp_value=1.5, clamp_count=cnt),
        "swiglu_bwd": lambda: tkq.swiglu_backward_and_per_token_cast(xg, dy),
    }
    exact = {"per_channel_t": oracle.per_channel_cast(xc, "e4m3", transpose=True, threads=THREADS),
             "per_block": oracle.per_block_cast(xb, "e4m3", threads=THREADS)}
    for name, op in ops.items():
        first = [t.clone() for t in op()]
        torch.cuda.synchronize()
        if name in exact:
            for a, e in zip(first, exact[name]):
                parity.assert_bit_exact(name, a.contiguous().view(torch.uint8).cpu().numpy(),
                                        np.ascontiguousarray(e).view(np.uint8))
        for _ in range(60):
            cur = op()
            torch.cuda.synchronize()
            for a, b in zip(first, cur):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{name} changed"
        cb_first = tkq.cast_back(first[0], first[1],
                                 group_size=(128, 128) if name == "per_block" else
                                 ((128, 1) if name == "per_channel" else (1, 128)),
                                 out_dtype=torch.bfloat16) if name in ("per_block", "per_channel") else None
        if cb_first is not None:
            for _ in range(20):
                again = tkq.cast_back(first[0], first[1],
                                      group_size=(128, 128) if name == "per_block" else (128, 1),
                                      out_dtype=torch.bfloat16)
                assert torch.equal(cb_first.view(torch.uint8), again.view(torch.uint8))
    assert tkq.tkq_read_device_status() == 0
