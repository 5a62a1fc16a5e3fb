"""Comparison of the CUDA path's outputs with the oracle's.

Tolerances:
* plain cast: codes and scales bit-exact;
* SwiGLU paths (y depends on the exp implementation, which differs between the
  CUDA math library and the oracle's correctly rounded exp): scales within
  1e-6 relative, codes within one FP8 step, at most 1e-4 of the codes differing.
  "One step" means adjacent in the ordered list of FP8 values, +0 and -0 equal.
"""
from __future__ import annotations

import numpy as np

SCALE_RTOL = 1e-6
CODE_MAX_STEP = 1
CODE_MAX_FRAC = 1e-4


def code_ordinal(codes: np.ndarray) -> np.ndarray:
    """Position of each FP8 code in the ordered list of values (finite codes):
    the magnitude bits give the order within a sign, negative codes count down,
    and both zeros map to 0."""
    c = np.asarray(codes).view(np.uint8).astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def assert_bit_exact(name: str, got: np.ndarray, exp: np.ndarray):
    got = np.ascontiguousarray(got)
    exp = np.ascontiguousarray(exp)
    assert got.shape == exp.shape, f"{name}: shape {got.shape} != {exp.shape}"
    gv = got.view(np.uint8 if got.dtype.itemsize == 1 else np.uint32)
    ev = exp.view(np.uint8 if exp.dtype.itemsize == 1 else np.uint32)
    bad = np.nonzero(gv.ravel() != ev.ravel())[0]
    assert bad.size == 0, (f"{name}: {bad.size} of {gv.size} differ; first at flat index "
                           f"{bad[:8].tolist()}: got {gv.ravel()[bad[:8]].tolist()} "
                           f"expected {ev.ravel()[bad[:8]].tolist()}")


def scale_rel_err(got: np.ndarray, exp: np.ndarray) -> float:
    g = np.asarray(got, np.float64)
    e = np.asarray(exp, np.float64)
    assert g.shape == e.shape
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - e) / np.abs(e)))


def assert_scales_close(name: str, got, exp, rtol=SCALE_RTOL):
    err = scale_rel_err(got, exp)
    assert err <= rtol, f"{name}: scale relative error {err:.3g} > {rtol:g}"


def code_diff_stats(got: np.ndarray, exp: np.ndarray):
    og = code_ordinal(got)
    oe = code_ordinal(exp)
    assert og.shape == oe.shape
    d = np.abs(og - oe)
    n = d.size
    return (int(d.max()) if n else 0), (int(np.count_nonzero(d)) if n else 0), n


def assert_codes_close(name: str, got, exp, max_step=CODE_MAX_STEP, max_frac=CODE_MAX_FRAC):
    mx, ndiff, n = code_diff_stats(got, exp)
    assert mx <= max_step, f"{name}: a code differs by {mx} steps (> {max_step})"
    assert ndiff <= max_frac * n, f"{name}: {ndiff} of {n} codes differ (> {max_frac:g})"
    return ndiff
