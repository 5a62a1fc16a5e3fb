"""The tie-aware code comparison used for the clamped SwiGLU must accept what
a few ulp of error in y can change and reject anything else (CPU only)."""
import numpy as np
import pytest

import oracle
from fp8_activation_quantization_gb300 import synth
from tests import parity


def _clamped(seed=81, T=256, H=256, c=1.0):
    x = synth.swiglu_bf16(seed, 82, T, H, gate_std=2.0)
    y, _ = oracle.swiglu_values(x, clamp=c)
    codes, sf = oracle.cast_rows_f32(y)
    return y, codes, sf


def test_accepts_tie_flips_from_a_few_ulp_of_error():
    y, codes, sf = _clamped()
    q = y / np.repeat(sf, 128, axis=1)
    flips = 0
    for k in (1, -1, 3, -3):
        yp = (y.astype(np.float64) * (1 + k * 2.0 ** -23)).astype(np.float32)
        # the perturbed values keep the oracle's scales (they are not the amax)
        cp = oracle.cast_rows_f32(yp)[0]
        flips += parity.assert_codes_differ_only_at_ties("perturbed", cp, codes, q, "e4m3")
    assert flips > 0          # clamping does create exact ties


def test_rejects_a_flip_away_from_a_tie():
    y, codes, sf = _clamped()
    q = y / np.repeat(sf, 128, axis=1)
    bad = codes.copy()
    vals = parity.fp8_values(codes, "e4m3")
    mid_dist = np.abs(q - np.round(q))      # any element not at a tie will do
    i, j = np.unravel_index(np.argmax((np.abs(vals) > 1) * mid_dist), codes.shape)
    bad[i, j] = (int(bad[i, j]) + 1) & 0xFF if bad[i, j] & 0x7F < 0x7E else bad[i, j] - 1
    with pytest.raises(AssertionError):
        parity.assert_codes_differ_only_at_ties("planted", bad, codes, q, "e4m3")


def test_rejects_two_step_differences():
    y, codes, sf = _clamped()
    q = y / np.repeat(sf, 128, axis=1)
    bad = codes.copy()
    k = np.nonzero((codes & 0x7F) > 4)
    bad[k[0][0], k[1][0]] -= 2
    with pytest.raises(AssertionError):
        parity.assert_codes_differ_only_at_ties("planted", bad, codes, q, "e4m3")
