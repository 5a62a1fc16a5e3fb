"""The per-token cast of fp32 inputs (through the C ABI) against the oracle's
fp32 row cast: codes and scales bit-exact.  The exhaustive test runs every
finite binary32 value of magnitude <= fmt_max through the kernel's hardware
conversion (in groups whose first element is fmt_max, so s = 1 exactly and each
code is the encoding of the value itself) and compares it with the oracle's
encoder.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq
from tests import parity
from tests.test_gpu_parity import Guarded, stream_of

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))
FMAX_BITS = {"e4m3": 0x43E00000, "e5m2": 0x47600000}   # 448.0f, 57344.0f


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def run_f32(y, fmt, dev, sf_flags=0):
    T, C = y.shape
    yd = torch.from_numpy(np.ascontiguousarray(y, np.float32)).to(dev)
    out = Guarded(T * C, dev)
    sf = Guarded(tkq.tkq_sf_bytes(T, C // 128, sf_flags), dev)
    st = tkq.tkq_per_token_cast_f32(ctypes.c_void_p(yd.data_ptr()), out.ptr, sf.ptr, T, C, 128,
                                    oracle.FMT[fmt], sf_flags, stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    return out.data().reshape(T, C), sf.data()


def f32_inputs(T, C, seed):
    """Magnitudes log-uniform over 2^-140 .. 2^20 (subnormals included),
    random signs, a zero row and a row of signed zeros."""
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-140.0, 20.0, (T, C)))
    y = (mag * rng.choice([-1.0, 1.0], (T, C))).astype(np.float32)
    if T > 2:
        y[1] = 0.0
        y[2] = -0.0
    return y


@pytest.mark.parametrize("T", [1, 7, 129, 1031])
@pytest.mark.parametrize("C", [128, 384, 2048])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_f32_cast_bit_exact(cuda_device, T, C, fmt):
    y = f32_inputs(T, C, T * 7 + C)
    codes, sf = run_f32(y, fmt, cuda_device)
    e_codes, e_sf = oracle.cast_rows_f32(y, fmt)
    parity.assert_bit_exact("sf", sf.view(np.float32).reshape(T, C // 128), e_sf)
    parity.assert_bit_exact("codes", codes, e_codes)


@pytest.mark.parametrize("flags", [1, 2, 4, 6])
def test_f32_cast_sf_layouts(cuda_device, flags):
    T, C = 301, 896
    y = f32_inputs(T, C, 91)
    codes, sf = run_f32(y, "e4m3", cuda_device, sf_flags=flags)
    e_codes, e_sf = oracle.cast_rows_f32_ex(y, "e4m3", flags=flags)
    parity.assert_bit_exact("codes", codes, e_codes)
    parity.assert_bit_exact("sf", sf.view(np.uint8), np.ascontiguousarray(e_sf).view(np.uint8).ravel())


def test_f32_tensor_api(cuda_device):
    y = f32_inputs(64, 256, 92)
    yd = torch.from_numpy(y).to(cuda_device)
    q, s = tkq.per_token_cast(yd, "e5m2")
    e_codes, e_sf = oracle.cast_rows_f32(y, "e5m2")
    assert q.dtype == torch.float8_e5m2 and s.shape == (64, 2)
    parity.assert_bit_exact("codes", q.view(torch.uint8).cpu().numpy(), e_codes)
    parity.assert_bit_exact("sf", s.cpu().numpy(), e_sf)


def _oracle_encode(vals: np.ndarray, fmt: str) -> np.ndarray:
    out = np.empty(vals.shape, np.uint8)
    parts = np.array_split(np.arange(vals.size), THREADS)

    def body(ix):
        if ix.size:
            out[ix[0]:ix[-1] + 1] = oracle.fp8_encode_array(vals[ix[0]:ix[-1] + 1], fmt)

    with ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(body, parts))
    return out


@pytest.mark.slow
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encoder_on_every_value_up_to_fmt_max(cuda_device, fmt):
    dev = cuda_device
    groups = 1 << 21                         # groups per launch: 1 GB of fp32 input
    per = 127 * groups                       # swept values per launch
    top = FMAX_BITS[fmt]                     # bit patterns 0 .. top are the values 0 .. fmt_max
    fmax = np.uint32(top).view(np.float32)
    checked = 0
    for sign in (0, 0x80000000):
        for start in range(0, top + 1, per):
            n = min(per, top + 1 - start)
            g = -(-n // 127)
            bits = torch.arange(start, start + g * 127, dtype=torch.int64, device=dev)
            bits = torch.clamp(bits, max=top)              # the tail repeats fmt_max
            if sign:
                bits = bits - (1 << 31)                    # 0x80000000 | b as a signed int32
            x = torch.empty((g, 128), dtype=torch.int32, device=dev)
            x[:, 0] = int(top)                             # the group leader: s = 1
            x[:, 1:] = bits.to(torch.int32).view(g, 127)
            x = x.view(torch.float32).view(-1, 2048) if g % 16 == 0 else x.view(torch.float32)
            T, C = x.shape
            out = torch.empty((T, C), dtype=torch.uint8, device=dev)
            sf = torch.empty((T, C // 128), dtype=torch.float32, device=dev)
            st = tkq.tkq_per_token_cast_f32(ctypes.c_void_p(x.data_ptr()),
                                            ctypes.c_void_p(out.data_ptr()),
                                            ctypes.c_void_p(sf.data_ptr()), T, C, 128,
                                            oracle.FMT[fmt], 0, stream_of(dev))
            assert st == 0, tkq.tkq_status_string(st)
            codes = out.view(g, 128).cpu().numpy()
            assert torch.all(sf == 1.0), "a group scale is not exactly 1"
            vals = x.view(g, 128)[:, 1:].cpu().numpy().ravel()
            got = codes[:, 1:].ravel()
            exp = _oracle_encode(vals, fmt)
            bad = np.nonzero(got != exp)[0]
            assert bad.size == 0, (f"{fmt}: {bad.size} codes differ, first value "
                                   f"{vals[bad[0]]!r} (bits {vals[bad[0]:bad[0]+1].view(np.uint32)[0]:#x}) "
                                   f"got {got[bad[0]]:#x} expected {exp[bad[0]]:#x}")
            lead = oracle.fp8_encode(float(fmax), fmt)
            assert np.all(codes[:, 0] == lead)
            checked += n
            del x, out, sf, bits
    assert checked == 2 * (top + 1)
