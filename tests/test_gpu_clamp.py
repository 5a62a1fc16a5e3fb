"""Parity of the clamped SwiGLU casts (through the C ABI) with the oracle.

Scales within 1e-6 relative; codes equal except by one FP8 step where the
oracle's quotient y / s lies at an FP8 rounding tie (clamping makes such ties
common: see parity.assert_codes_differ_only_at_ties); the clamp count is an
integer decided by exact comparisons of bf16 inputs with the bound, so it must
equal the oracle's count exactly.

For a bound that is itself a bf16 value the clamp of a bf16 input is again a
bf16 value, so the clamped cast must quantize exactly the kernels' own y of the
input clipped on the host (tkq_swiglu_values): its codes and scales then equal
bit for bit the oracle's reading of that y (the product by the rounded
reciprocal of the scale, which the SwiGLU kernels compute), with no exception
at ties.
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


def q_rows(x, w, clamp, sf):
    """The oracle's quotients y / s of the row cast."""
    y, _ = oracle.swiglu_values(x, w, THREADS, clamp=clamp)
    return y / np.repeat(sf, 128, axis=1)


def q_cols(x, w, clamp, sf_t):
    """The oracle's quotients y[t, c] / s_t of the transposed cast, as [H, T]."""
    y, _ = oracle.swiglu_values(x, w, THREADS, clamp=clamp)
    return y.T / np.repeat(sf_t, 128, axis=1)


def run_clamp(x_bits, w, fmt, clamp, dev, transposed=False, count=None, sf_flags=0):
    """One clamped launch; returns the outputs and the counter's value (the
    counter starts at `count` if given, else at 0)."""
    T, H2 = x_bits.shape
    H = H2 // 2
    xd = to_dev_bf16(x_bits, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    wp = None if wd is None else ctypes.c_void_p(wd.data_ptr())
    cnt = torch.full((1,), 0 if count is None else count, dtype=torch.int64, device=dev)
    out = Guarded(T * H, dev)
    f = oracle.FMT[fmt]
    cp = ctypes.c_void_p(cnt.data_ptr())
    if not transposed:
        sf = Guarded(tkq.tkq_sf_bytes(T, H // 128, sf_flags), dev)
        st = tkq.tkq_swiglu_cast_clamp(ctypes.c_void_p(xd.data_ptr()), wp, out.ptr, sf.ptr, T, H,
                                       128, f, sf_flags, clamp, cp, stream_of(dev))
        assert st == 0, tkq.tkq_status_string(st)
        torch.cuda.synchronize()
        out.check_guards("out")
        sf.check_guards("sf")
        return out.data().reshape(T, H), sf.data(), int(cnt.item())
    sf = Guarded(T * (H // 128) * 4, dev)
    out_t = Guarded(T * H, dev)
    sf_t = Guarded(H * (T // 128) * 4, dev)
    st = tkq.tkq_swiglu_cast_t_clamp(ctypes.c_void_p(xd.data_ptr()), wp, out.ptr, sf.ptr,
                                     out_t.ptr, sf_t.ptr, T, H, 128, f, 0, clamp, cp,
                                     stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    for g, n in ((out, "out"), (sf, "sf"), (out_t, "out_t"), (sf_t, "sf_t")):
        g.check_guards(n)
    return (out.data().reshape(T, H), sf.data().view(np.float32).reshape(T, H // 128),
            out_t.data().reshape(H, T), sf_t.data().view(np.float32).reshape(H, T // 128),
            int(cnt.item()))


# Bounds that are bf16 values take the packed-bf16 clamp; 0.7 and 2.9 are not
# bf16 values and take the fp32 clamp.
@pytest.mark.parametrize("clamp", [0.5, 3.0, 0.7, 2.9])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("T,H", [(1, 128), (1031, 384)])
def test_clamped_swiglu_cast(cuda_device, swiglu_kernel, clamp, weighted, fmt, T, H):
    x = synth.swiglu_bf16(71, T + H, T, H, gate_std=2.0)
    w = synth.routing_weights(72, T, -(-T // 8))[:T] if weighted else None
    codes, sf_raw, n = run_clamp(x, w, fmt, clamp, cuda_device)
    e_codes, e_sf, e_n = oracle.swiglu_cast(x, w, fmt, threads=THREADS, clamp=clamp)
    assert n == e_n
    parity.assert_scales_close("sf", sf_raw.view(np.float32).reshape(T, H // 128), e_sf)
    parity.assert_codes_differ_only_at_ties("codes", codes, e_codes, q_rows(x, w, clamp, e_sf), fmt)


def test_clamped_swiglu_full_workload(cuda_device):
    d = synth.workload("swiglu")
    x = d["x"]
    T, H = x.shape[0], x.shape[1] // 2
    codes, sf_raw, n = run_clamp(x, None, "e4m3", 4.0, cuda_device)
    e_codes, e_sf, e_n = oracle.swiglu_cast(x, None, "e4m3", threads=THREADS, clamp=4.0)
    assert n == e_n and n > 0
    parity.assert_scales_close("sf", sf_raw.view(np.float32).reshape(T, H // 128), e_sf)
    parity.assert_codes_differ_only_at_ties("codes", codes, e_codes,
                                            q_rows(x, None, 4.0, e_sf), "e4m3")


def clip_on_host(x_bits, c):
    """The clamp applied to the bf16 input itself (c a bf16 value, > 0): gates
    to <= c, ups to [-c, c]; the results are bf16 values, returned as bits."""
    H = x_bits.shape[1] // 2
    v = synth.bf16_bits_to_f32(x_bits)
    v[:, :H] = np.minimum(v[:, :H], np.float32(c))
    v[:, H:] = np.clip(v[:, H:], np.float32(-c), np.float32(c))
    bits = np.ascontiguousarray((v.view(np.uint32) >> 16).astype(np.uint16))
    assert np.array_equal(synth.bf16_bits_to_f32(bits), v)   # exact: c is a bf16 value
    return bits


@pytest.mark.parametrize("clamp", [4.0, 0.5])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_clamped_casts_quantize_the_clipped_values(cuda_device, swiglu_kernel, clamp, weighted,
                                                   fmt):
    """With a bf16 bound, the clamped row cast and the clamped transposed cast
    quantize exactly the kernels' y of the host-clipped input: codes and
    scales, rows and columns, bit for bit against the oracle's reading of that
    y; the count is the number of values the clip changed."""
    T, H = 1024, 384
    x = synth.swiglu_bf16(81, 82, T, H, gate_std=2.0)
    w = synth.routing_weights(83, 84, T // 8) if weighted else None
    xc = clip_on_host(x, clamp)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).to(cuda_device)
    y = tkq.swiglu_values(to_dev_bf16(xc, cuda_device), wd).cpu().numpy()
    e_q, e_s = oracle.cast_rows_f32_ex(y, fmt, 128, oracle.Q_RECIPROCAL)
    changed = int(np.count_nonzero(xc != x))
    codes, sf_raw, n = run_clamp(x, w, fmt, clamp, cuda_device)
    assert n == changed > 0
    parity.assert_bit_exact("codes", codes, e_q)
    parity.assert_bit_exact("scales", sf_raw.view(np.float32).reshape(T, H // 128), e_s)
    o, s, ot, st, n_t = run_clamp(x, w, fmt, clamp, cuda_device, transposed=True)
    e_qt, e_st = oracle.cast_rows_f32_ex(np.ascontiguousarray(y.T), fmt, 128, oracle.Q_RECIPROCAL)
    assert n_t == changed
    parity.assert_bit_exact("rows", o, e_q)
    parity.assert_bit_exact("row scales", s, e_s)
    parity.assert_bit_exact("column codes", ot, e_qt)
    parity.assert_bit_exact("column scales", st, e_st)


def test_clamped_full_workload_quantizes_the_clipped_values(cuda_device):
    """The swiglu workload with c = 4 (about 2.3 % of the gates clipped) through
    the clamped transposed cast: rows and columns bit for bit against the
    oracle's reading of the kernels' y of the host-clipped input."""
    x = synth.workload("swiglu")["x"]
    xc = clip_on_host(x, 4.0)
    y = tkq.swiglu_values(to_dev_bf16(xc, cuda_device)).cpu().numpy()
    o, s, ot, st, n = run_clamp(x, None, "e4m3", 4.0, cuda_device, transposed=True)
    assert n == int(np.count_nonzero(xc != x))
    e_q, e_s = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.Q_RECIPROCAL, threads=THREADS)
    parity.assert_bit_exact("rows", o, e_q)
    parity.assert_bit_exact("row scales", s, e_s)
    del e_q, e_s
    e_qt, e_st = oracle.cast_rows_f32_ex(np.ascontiguousarray(y.T), "e4m3", 128,
                                         oracle.Q_RECIPROCAL, threads=THREADS)
    parity.assert_bit_exact("column codes", ot, e_qt)
    parity.assert_bit_exact("column scales", st, e_st)


@pytest.mark.parametrize("clamp", [2.0, 1.3])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("T,H", [(128, 128), (1024, 384)])
def test_clamped_swiglu_cast_t(cuda_device, clamp, weighted, T, H):
    x = synth.swiglu_bf16(73, T + H, T, H, gate_std=2.0)
    w = synth.routing_weights(74, T, T // 8) if weighted else None
    o, s, ot, st, n = run_clamp(x, w, "e4m3", clamp, cuda_device, transposed=True)
    eo, es, eot, est, e_n = oracle.swiglu_cast_t(x, w, "e4m3", threads=THREADS, clamp=clamp)
    assert n == e_n
    parity.assert_scales_close("sf", s, es)
    parity.assert_codes_differ_only_at_ties("codes", o, eo, q_rows(x, w, clamp, es), "e4m3")
    parity.assert_scales_close("sf_t", st, est)
    parity.assert_codes_differ_only_at_ties("codes_t", ot, eot, q_cols(x, w, clamp, est), "e4m3")
    # the row outputs equal the clamped row cast's bit for bit
    o2, s2, n2 = run_clamp(x, w, "e4m3", clamp, cuda_device)
    parity.assert_bit_exact("rows", o, o2)
    parity.assert_bit_exact("row scales", s, s2.view(np.float32).reshape(s.shape))
    assert n2 == n


def test_clamped_swiglu_cast_t_full_workload(cuda_device):
    x = synth.workload("swiglu")["x"]
    o, s, ot, st, n = run_clamp(x, None, "e4m3", 4.0, cuda_device, transposed=True)
    eo, es, eot, est, e_n = oracle.swiglu_cast_t(x, None, "e4m3", threads=THREADS, clamp=4.0)
    assert n == e_n and n > 0
    parity.assert_scales_close("sf_t", st, est)
    parity.assert_codes_differ_only_at_ties("codes_t", ot, eot, q_cols(x, None, 4.0, est), "e4m3")


def test_clamp_count_accumulates_and_null_counter_is_allowed(cuda_device, swiglu_kernel):
    x = synth.swiglu_bf16(75, 76, 512, 256, gate_std=2.0)
    _, _, n1 = run_clamp(x, None, "e4m3", 1.0, cuda_device)
    _, _, n2 = run_clamp(x, None, "e4m3", 1.0, cuda_device, count=n1)
    assert n1 > 0 and n2 == 2 * n1
    xd = to_dev_bf16(x, cuda_device)
    q, s = tkq.swiglu_forward_and_per_token_cast(xd, use_clamp=True, swiglu_clamp_value=1.0)
    c, _, _ = run_clamp(x, None, "e4m3", 1.0, cuda_device)
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), c)
    cnt = torch.zeros(1, dtype=torch.int64, device=cuda_device)
    tkq.swiglu_forward_and_per_token_cast(xd, use_clamp=True, swiglu_clamp_value=1.0,
                                          clamp_count=cnt, with_transpose=True)
    assert int(cnt.item()) == n1


def test_clamp_beyond_the_data_is_the_unclamped_cast(cuda_device, swiglu_kernel):
    x = synth.swiglu_bf16(77, 78, 300, 256)
    xd = to_dev_bf16(x, cuda_device)
    q0, s0 = tkq.swiglu_forward_and_per_token_cast(xd)
    q1, s1, n = run_clamp(x, None, "e4m3", 1e30, cuda_device)
    assert n == 0
    assert np.array_equal(q0.view(torch.uint8).cpu().numpy(), q1)
    assert np.array_equal(s0.cpu().numpy().view(np.uint32).ravel(), s1.view(np.uint32))


def test_clamp_with_column_major_scales(cuda_device, swiglu_kernel):
    """The clamp composes with a scale layout: column-major fp32 scales are the
    row-major scales of the same clamped launch, transposed (and padded)."""
    T, H = 301, 384
    x = synth.swiglu_bf16(79, 80, T, H, gate_std=2.0)
    c0, s0, n0 = run_clamp(x, None, "e4m3", 2.0, cuda_device)
    c1, s1, n1 = run_clamp(x, None, "e4m3", 2.0, cuda_device, sf_flags=tkq.SF_COL_MAJOR)
    T4 = (T + 3) // 4 * 4
    rm = s0.view(np.float32).reshape(T, H // 128)
    cm = s1.view(np.float32).reshape(H // 128, T4)
    assert n0 == n1 and np.array_equal(c0, c1)
    assert np.array_equal(cm[:, :T], rm.T) and np.all(cm[:, T:] == 0)


def _bf16_neighbours(c):
    """bf16 bit patterns at and around the bound c (> 0): the largest bf16
    value below c, c itself when it is a bf16 value, and the smallest above."""
    b = int(np.float32(c).view(np.uint32))
    lo = b >> 16
    if b & 0xFFFF:
        return [lo, lo + 1]
    return [lo - 1, lo, lo + 1]


# 2.0 and 448.0 are bf16 values (packed-bf16 clamp); 2.0 + 2^-20 and 0.3 are
# not (fp32 clamp).  NaN inputs are outside the contract and not drawn.
@pytest.mark.parametrize("clamp", [2.0, 448.0, 2.0 + 2.0 ** -20, 0.3])
@pytest.mark.parametrize("weighted", [False, True])
def test_clamp_at_special_values(cuda_device, swiglu_kernel, clamp, weighted):
    """Gates and ups drawn from infinities, the largest finite bf16, signed
    zeros, bf16 subnormals, and the bf16 values at and next to +-c: the count
    is exact and the outputs match the oracle (row and transposed casts)."""
    near = _bf16_neighbours(clamp)
    subnormals = [0x0001, 0x8001, 0x007F, 0x807F]        # must pass the clamp unchanged
    gates = np.array([0x7F80, 0x7F7F, 0x3F80, 0x0000, 0x8000, 0xC0A0, 0xC2C8]
                     + subnormals + near + [n | 0x8000 for n in near], np.uint16)
    ups = np.array([0x7F80, 0xFF80, 0x7F7F, 0xFF7F, 0x0000, 0x8000, 0x3F00]
                   + subnormals + near + [n | 0x8000 for n in near], np.uint16)
    rng = np.random.default_rng(int(clamp * 1000) + weighted)
    T, H = 256, 256
    x = np.concatenate([rng.choice(gates, (T, H)), rng.choice(ups, (T, H))], axis=1)
    x = np.ascontiguousarray(x.astype(np.uint16))
    w = synth.routing_weights(77, T, T // 8) if weighted else None
    codes, sf_raw, n = run_clamp(x, w, "e4m3", clamp, cuda_device)
    e_codes, e_sf, e_n = oracle.swiglu_cast(x, w, "e4m3", threads=THREADS, clamp=clamp)
    assert n == e_n > 0
    parity.assert_scales_close("sf", sf_raw.view(np.float32).reshape(T, H // 128), e_sf)
    parity.assert_codes_differ_only_at_ties("codes", codes, e_codes, q_rows(x, w, clamp, e_sf),
                                            "e4m3")
    o, s, ot, st, n_t = run_clamp(x, w, "e4m3", clamp, cuda_device, transposed=True)
    eo, es, eot, est, _ = oracle.swiglu_cast_t(x, w, "e4m3", threads=THREADS, clamp=clamp)
    assert n_t == e_n
    parity.assert_bit_exact("rows", o, codes)
    parity.assert_scales_close("sf_t", st, est)
    parity.assert_codes_differ_only_at_ties("codes_t", ot, eot, q_cols(x, w, clamp, est), "e4m3")
