"""The SwiGLU values the casts quantize, checked value by value.

tkq_swiglu_values writes the fp32 y = silu(g) * u [* w] that the SwiGLU casts
compute (the SM's ex2 / rcp on packed pairs).  Against a binary64 evaluation
each value must lie within the bound derived for that evaluation:
exp(-g) = 2^(-g log2 e) carries about (1.04 |t| + 2) ulp of relative error
(t = g log2 e, the rounded product's error amplified by the exponential), which
reaches y scaled by e / (1 + e); the rounded add, the approximate reciprocal
and the two or three products add at most 4 ulp more.  Values whose binary64
magnitude is tiny are compared with an absolute floor of |g u w| 2^-125
(rcp.approx.ftz flushes 1 / (1 + e) to zero below 2^-126, i.e. for g < -87.3,
where y is then 0; the codes there are a signed zero either way).

Then the casts are shown to quantize exactly these values: the SwiGLU cast's
scales equal bit for bit the oracle's scale rule applied to the diagnostic y,
and its codes equal the oracle's codes of that y except at FP8 ties (and bit
for bit the codes of the oracle's reciprocal-multiply reading, the product by
fl32(1 / s) that the kernels compute), with and without scale layouts.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests import parity
from tests.test_gpu_parity import to_dev_bf16

pytestmark = pytest.mark.gpu

ULP = 2.0 ** -24
LOG2E = 1.4426950408889634


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def reference_and_bound(g, u, w):
    """binary64 y and the allowed absolute error per element."""
    g = g.astype(np.float64)
    u = u.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        e = np.exp(-g)
        y = g / (1.0 + e) * u * w
        frac = np.where(np.isinf(e), 1.0, e / (1.0 + e))
    t = np.abs(g) * LOG2E
    rel = ((1.04 * t + 2.0) * frac + 4.0) * ULP
    # absolute floor: rcp.approx.ftz flushes 1 / (1 + e) to zero once it is
    # below 2^-126 (g < -87.3), where the exact |y| is at most |g u w| 2^-126
    floor = 2.0 ** -125 * np.maximum(1.0, np.abs(g * u * w))
    return y, rel * np.abs(y) + floor


def all_finite_bf16_gates():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = synth.bf16_bits_to_f32(bits)
    return bits[np.isfinite(v)]


@pytest.mark.parametrize("u_val,w_val", [(1.0, None), (-0.75, 0.37)])
def test_every_bf16_gate_within_the_bound(cuda_device, u_val, w_val):
    gates = all_finite_bf16_gates()
    H = 1024
    n = -(-gates.size // H) * H
    gbits = np.resize(gates, n).reshape(-1, H)            # pad by repeating
    T = gbits.shape[0]
    ubits = np.full((T, H), synth.f32_to_bf16_bits(np.float32(u_val)), np.uint16)
    x = np.ascontiguousarray(np.concatenate([gbits, ubits], axis=1))
    w = None if w_val is None else np.full(T, w_val, np.float32)
    xd = to_dev_bf16(x, cuda_device)
    wd = None if w is None else torch.from_numpy(w).to(cuda_device)
    y = tkq.swiglu_values(xd, wd).cpu().numpy().astype(np.float64)
    g = synth.bf16_bits_to_f32(gbits)
    u = synth.bf16_bits_to_f32(ubits)
    ref, tol = reference_and_bound(g, u, 1.0 if w is None else np.float64(np.float32(w_val)))
    err = np.abs(y - ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} values outside the bound; worst gate "
                           f"{g.ravel()[np.argmax(err / tol)]!r}: y {y.ravel()[np.argmax(err / tol)]!r} "
                           f"vs {ref.ravel()[np.argmax(err / tol)]!r}")


def test_random_values_within_the_bound(cuda_device):
    rng = np.random.default_rng(5)
    T, H = 4096, 1024
    g = (rng.standard_normal((T, H)) * 4.0).astype(np.float32)
    u = rng.standard_normal((T, H)).astype(np.float32)
    w = rng.uniform(0.01, 1.0, T).astype(np.float32)
    x = np.concatenate([synth.f32_to_bf16_bits(g), synth.f32_to_bf16_bits(u)], axis=1)
    x = np.ascontiguousarray(x)
    y = tkq.swiglu_values(to_dev_bf16(x, cuda_device),
                          torch.from_numpy(w).to(cuda_device)).cpu().numpy().astype(np.float64)
    gb = synth.bf16_bits_to_f32(x[:, :H])
    ub = synth.bf16_bits_to_f32(x[:, H:])
    ref, tol = reference_and_bound(gb, ub, w.astype(np.float64)[:, None])
    # the weight multiply is one more rounded product
    tol = tol + ULP * np.abs(ref)
    assert np.all(np.abs(y - ref) <= tol)


@pytest.mark.parametrize("weighted", [False, True])
def test_casts_quantize_these_values(cuda_device, swiglu_kernel, weighted):
    """Scales of the SwiGLU cast = the oracle's scale rule on the diagnostic y
    (bit for bit); codes = the oracle's codes of that y except at FP8 ties
    (the cast multiplies by the rounded reciprocal, the oracle divides)."""
    d = synth.workload("swiglu_moe", rows=4096)
    x = np.ascontiguousarray(d["x"][:, np.r_[0:1024, 2048:3072]])
    w = d["w"] if weighted else None
    xd = to_dev_bf16(x, cuda_device)
    wd = None if w is None else torch.from_numpy(w).to(cuda_device)
    y = tkq.swiglu_values(xd, wd).cpu().numpy()
    q, s = tkq.swiglu_forward_and_per_token_cast(xd, topk_weights=wd)
    e_q, e_s = oracle.cast_rows_f32(y, "e4m3")
    parity.assert_bit_exact("scales", s.cpu().numpy(), e_s)
    parity.assert_codes_differ_only_at_ties("codes", q.view(torch.uint8).cpu().numpy(), e_q,
                                            y / np.repeat(e_s, 128, axis=1), "e4m3")
    # the codes are exactly the reciprocal-multiply reading of y
    e_qr, _ = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.Q_RECIPROCAL)
    parity.assert_bit_exact("codes (reciprocal reading)", q.view(torch.uint8).cpu().numpy(), e_qr)
    # the transposed kernel quantizes the same y as well
    q2, s2, qt, st = tkq.swiglu_forward_and_per_token_cast(xd, topk_weights=wd, with_transpose=True)
    e_qt, e_st = oracle.cast_cols_f32(y, "e4m3")
    parity.assert_bit_exact("column scales", st.cpu().numpy(), e_st)
    parity.assert_codes_differ_only_at_ties("column codes", qt.view(torch.uint8).cpu().numpy(), e_qt,
                                            y.T / np.repeat(e_st, 128, axis=1), "e4m3")
    e_qtr, _ = oracle.cast_rows_f32_ex(np.ascontiguousarray(y.T), "e4m3", 128, oracle.Q_RECIPROCAL)
    parity.assert_bit_exact("column codes (reciprocal reading)",
                            qt.view(torch.uint8).cpu().numpy(), e_qtr)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["swiglu_moe", "swiglu_t"])
def test_full_workloads_quantize_these_values(cuda_device, name):
    """At the full sizes of the weighted SwiGLU workload and of the transposed
    workload (the benchmark's step): every row scale, and for the transposed
    cast every column scale, equals bit for bit the oracle's scale rule applied
    to the kernels' own y; every code equals the oracle's code of that y except
    at FP8 ties, and equals bit for bit the code of its reciprocal-multiply
    reading (the product by fl32(1 / s), which is what the kernels compute)."""
    d = synth.workload(name)
    x, w = d["x"], d.get("w")
    xd = to_dev_bf16(x, cuda_device)
    wd = None if w is None else torch.from_numpy(w).to(cuda_device)
    y = tkq.swiglu_values(xd, wd).cpu().numpy()
    if name == "swiglu_t":
        q, s, qt, st = tkq.swiglu_forward_and_per_token_cast(xd, with_transpose=True)
    else:
        q, s = tkq.swiglu_forward_and_per_token_cast(xd, topk_weights=wd)
    del xd
    e_q, e_s = oracle.cast_rows_f32(y, "e4m3")
    parity.assert_bit_exact("row scales", s.cpu().numpy(), e_s)
    parity.assert_codes_differ_only_at_ties("row codes", q.view(torch.uint8).cpu().numpy(), e_q,
                                            y / np.repeat(e_s, 128, axis=1), "e4m3")
    e_qr, _ = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.Q_RECIPROCAL, threads=16)
    parity.assert_bit_exact("row codes (reciprocal reading)", q.view(torch.uint8).cpu().numpy(),
                            e_qr)
    del e_q, e_s, e_qr, q, s
    if name == "swiglu_t":
        e_qt, e_st = oracle.cast_cols_f32(y, "e4m3")
        parity.assert_bit_exact("column scales", st.cpu().numpy(), e_st)
        parity.assert_codes_differ_only_at_ties(
            "column codes", qt.view(torch.uint8).cpu().numpy(), e_qt,
            y.T / np.repeat(e_st, 128, axis=1), "e4m3")
        del e_qt
        e_qtr, _ = oracle.cast_rows_f32_ex(np.ascontiguousarray(y.T), "e4m3", 128,
                                           oracle.Q_RECIPROCAL, threads=16)
        parity.assert_bit_exact("column codes (reciprocal reading)",
                                qt.view(torch.uint8).cpu().numpy(), e_qtr)


def _raw(t):
    return np.ascontiguousarray(t.contiguous().view(torch.uint8).cpu().numpy()).ravel()


@pytest.mark.parametrize("flags,fmt", [(1, "e4m3"), (2, "e4m3"), (4, "e4m3"), (6, "e5m2"),
                                       (7, "e4m3"), (8, "e5m2")])
def test_transposed_cast_layouts_quantize_these_values(cuda_device, flags, fmt):
    """The transposed cast with a scale layout: its row codes and scales, and
    its column codes and scales (an [H, T/128] matrix in the same layout),
    equal bit for bit the oracle's reciprocal-multiply reading of the kernels'
    own y in that layout (rows of y, rows of y transposed); the row outputs
    equal the row cast's with the same flags.  T = 384 and H = 640 leave
    partly used packed words on both scale matrices."""
    T, H = 384, 640
    x = synth.swiglu_bf16(61, 3, T, H, gate_std=2.0)
    w = synth.routing_weights(62, 4, T // 8)
    xd = to_dev_bf16(x, cuda_device)
    wd = torch.from_numpy(w).to(cuda_device)
    opts = dict(round_sf=bool(flags & 1), use_packed_ue8m0=bool(flags & 2),
                use_tma_aligned_col_major_sf=bool(flags & 4))
    y = tkq.swiglu_values(xd, wd).cpu().numpy()
    q, s, qt, st = tkq.swiglu_forward_and_per_token_cast(xd, fmt, topk_weights=wd,
                                                         with_transpose=True, **opts)
    e_q, e_s = oracle.cast_rows_f32_ex(y, fmt, 128, flags | oracle.Q_RECIPROCAL)
    e_qt, e_st = oracle.cast_rows_f32_ex(np.ascontiguousarray(y.T), fmt, 128,
                                         flags | oracle.Q_RECIPROCAL)
    parity.assert_bit_exact("row codes", q.view(torch.uint8).cpu().numpy(), e_q)
    parity.assert_bit_exact("row scales (layout bytes)", _raw(s), e_s.view(np.uint8).ravel())
    parity.assert_bit_exact("column codes", qt.view(torch.uint8).cpu().numpy(), e_qt)
    parity.assert_bit_exact("column scales (layout bytes)", _raw(st), e_st.view(np.uint8).ravel())
    q2, s2 = tkq.swiglu_forward_and_per_token_cast(xd, fmt, topk_weights=wd, **opts)
    assert torch.equal(q.view(torch.uint8), q2.view(torch.uint8))
    assert np.array_equal(_raw(s), _raw(s2))
