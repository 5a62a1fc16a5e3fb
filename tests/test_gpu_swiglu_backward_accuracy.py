"""The SwiGLU gradients the backward cast quantizes, checked value by value.

tkq_swiglu_backward_values writes the fp32 [dg | du] that the backward cast
computes (swiglu_grad2: the SM's ex2 / rcp on packed pairs, then the weight
product).  Against a binary64 evaluation of
    dg = d u S (1 + g O) w,   du = d g S w,   S = 1 / (1 + E), O = E S, E = exp(-g)
each value must lie within the bound derived from the steps the kernel takes
(U = 2^-24, binary32 rounding to nearest):
    e      = ex2(fl(-g log2 e))      relative error e_E = (1.04 |g| log2 e + 2) U
                                     (as for the forward values)
    sigma  = rcp(fl(1 + e))          e_S = O e_E + U (add) + 2 U (rcp, 1 ulp)
    1 - s  = min(fl(e sigma), 1)     e_O = e_E + e_S + U
    f      = fma(g, 1 - s, 1)        absolute |g| O e_O + U |F|,  F = 1 + g O
    dsilu  = fl(sigma f)             absolute S |df| + |S F| (e_S + U)
    dg     = fl(fl(d u) dsilu) [w]   absolute |d u w| |d dsilu| + 3 U |dg|
    du     = fl(d fl(g sigma)) [w]   relative e_S + 3 U
with 1 % on top for second-order terms.  Where sigma is below the smallest
normal binary32 (E > 2^125.9, i.e. g < -87.3) rcp flushes it to zero and both
computed gradients are 0: there the error is the exact value itself, at most
|d u w| S (1 + |g|) (an exponent clamped at 126 instead would leave
2^-126 |1 + g| |d u w|, which this rejects below g = -89).  Where e is below
the smallest normal (g > 87.3) it flushes to zero; the exact values differ
from the computed ones by less than 2^-126 (1 + |g|) relative, far inside the
rounding terms.

Then the backward cast is shown to quantize exactly these values: its scales
equal bit for bit the oracle's scale rule applied to them, and its codes the
oracle's codes except at FP8 ties, on random shapes and at full size.
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

U = 2.0 ** -24
LOG2E = 1.4426950408889634
FLUSH_E = 2.0 ** 125.9


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def reference_and_bounds(g, u, d, w):
    """binary64 (dg, du) and the allowed absolute error of each."""
    g, u, d = (np.asarray(a, np.float64) for a in (g, u, d))
    w = np.asarray(w, np.float64)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore", under="ignore"):
        E = np.exp(-g)
        S = 1.0 / (1.0 + E)
        O = np.where(np.isinf(E), 1.0, E * S)
        F = 1.0 + g * O
        DS = S * F
        DG = d * u * DS * w
        DU = d * g * S * w
        e_E = (1.04 * np.abs(g) * LOG2E + 2.0) * U
        e_S = O * e_E + 3.0 * U
        e_O = e_E + e_S + U
        df = np.abs(g) * O * e_O + U * np.abs(F)
        dds = S * df + np.abs(DS) * (e_S + U)
        duw = np.abs(d * u * w)
        tol_dg = 1.01 * (duw * dds + 3.0 * U * np.abs(DG))
        tol_du = 1.01 * np.abs(DU) * (e_S + 3.0 * U)
        flushed = E > FLUSH_E
        tol_dg = np.where(flushed, tol_dg + 2.0 * np.abs(DG) + 2.0 * duw * S * (1.0 + np.abs(g)),
                          tol_dg)
        tol_du = np.where(flushed, tol_du + 2.0 * np.abs(DU), tol_du)
    return DG, DU, tol_dg + 2.0 ** -140, tol_du + 2.0 ** -140


def _values(x_bits, dy_bits, w, dev):
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    y = tkq.swiglu_backward_values(to_dev_bf16(x_bits, dev), to_dev_bf16(dy_bits, dev), wd)
    return y.cpu().numpy()


def _check(name, got, ref, tol):
    err = np.abs(got.astype(np.float64) - ref)
    bad = ~(err <= tol)
    if bad.any():
        k = np.argmax(np.where(bad, err / np.maximum(tol, 1e-300), 0.0))
        raise AssertionError(f"{name}: {int(bad.sum())} values outside the bound; worst at flat "
                             f"index {k}: got {got.ravel()[k]!r}, binary64 {ref.ravel()[k]!r}, "
                             f"bound {tol.ravel()[k]:.3g}")


@pytest.mark.parametrize("u_val,d_val,w_val", [(1.0, 1.0, None), (-0.75, 0.8125, 0.37)])
def test_every_bf16_gate_within_the_bound(cuda_device, u_val, d_val, w_val):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    gates = bits[np.isfinite(synth.bf16_bits_to_f32(bits))]
    H = 1024
    gbits = np.resize(gates, -(-gates.size // H) * H).reshape(-1, H)   # pad by repeating
    T = gbits.shape[0]
    ubits = np.full((T, H), synth.f32_to_bf16_bits(np.float32(u_val)), np.uint16)
    dbits = np.full((T, H), synth.f32_to_bf16_bits(np.float32(d_val)), np.uint16)
    x = np.ascontiguousarray(np.concatenate([gbits, ubits], axis=1))
    w = None if w_val is None else np.full(T, w_val, np.float32)
    y = _values(x, dbits, w, cuda_device)
    g = synth.bf16_bits_to_f32(gbits)
    wt = 1.0 if w is None else np.float64(np.float32(w_val))
    DG, DU, tg, tu = reference_and_bounds(g, np.float32(u_val), np.float32(d_val), wt)
    _check("dg", y[:, :H], DG, tg)
    _check("du", y[:, H:], DU, tu)
    # the overflow region: every gate below -89 gives exactly zero gradients
    far = g < -89.0
    assert far.any() and np.all(y[:, :H][far] == 0) and np.all(y[:, H:][far] == 0)


def test_random_values_within_the_bound(cuda_device):
    rng = np.random.default_rng(11)
    T, H = 2048, 1024
    g = (rng.standard_normal((T, H)) * 4.0).astype(np.float32)
    g[:, :16] = rng.uniform(-120.0, 120.0, (T, 16)).astype(np.float32)   # both flush regions
    u = rng.standard_normal((T, H)).astype(np.float32)
    dd = rng.standard_normal((T, H)).astype(np.float32)
    w = rng.uniform(0.01, 1.0, T).astype(np.float32)
    x = np.ascontiguousarray(np.concatenate([synth.f32_to_bf16_bits(g), synth.f32_to_bf16_bits(u)],
                                            axis=1))
    dbits = synth.f32_to_bf16_bits(dd)
    y = _values(x, dbits, w, cuda_device)
    DG, DU, tg, tu = reference_and_bounds(synth.bf16_bits_to_f32(x[:, :H]),
                                          synth.bf16_bits_to_f32(x[:, H:]),
                                          synth.bf16_bits_to_f32(dbits), w[:, None])
    _check("dg", y[:, :H], DG, tg)
    _check("du", y[:, H:], DU, tu)


def _cast_matches_values(x, dy, w, dev, fmt="e4m3"):
    """The backward cast's scales = the oracle's scale rule on the diagnostic
    values (bit for bit); its codes = the oracle's codes of them except at ties,
    and bit for bit those of the reciprocal-multiply reading."""
    xd, dyd = to_dev_bf16(x, dev), to_dev_bf16(dy, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    y = tkq.swiglu_backward_values(xd, dyd, wd).cpu().numpy()
    q, s = tkq.swiglu_backward_and_per_token_cast(xd, dyd, fmt, topk_weights=wd)
    e_q, e_s = oracle.cast_rows_f32(y, fmt)
    parity.assert_bit_exact("scales", s.cpu().numpy(), e_s)
    parity.assert_codes_differ_only_at_ties("codes", q.view(torch.uint8).cpu().numpy(), e_q,
                                            y / np.repeat(e_s, 128, axis=1), fmt)
    e_qr, _ = oracle.cast_rows_f32_ex(y, fmt, 128, oracle.Q_RECIPROCAL, threads=16)
    parity.assert_bit_exact("codes (reciprocal reading)", q.view(torch.uint8).cpu().numpy(), e_qr)


@pytest.mark.parametrize("T,H,weighted,fmt", [(1, 128, False, "e4m3"), (129, 384, True, "e4m3"),
                                              (1031, 256, True, "e5m2")])
def test_cast_quantizes_these_values(cuda_device, T, H, weighted, fmt):
    x = synth.swiglu_bf16(T, H, T, H, gate_std=3.0)
    dy = synth.normal_bf16(T + 1, H, T, H)
    w = synth.routing_weights(T, 2, -(-T // 8))[:T] if weighted else None
    _cast_matches_values(x, dy, w, cuda_device, fmt)


@pytest.mark.slow
def test_full_workload_cast_quantizes_these_values(cuda_device):
    d = synth.workload("swiglu_bwd")
    _cast_matches_values(d["x"], d["dy"], d["w"], cuda_device)
