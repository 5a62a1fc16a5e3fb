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


def fp8_values(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Values of FP8 codes (torch's float8 dtypes decode them)."""
    import torch
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    c = torch.from_numpy(np.ascontiguousarray(codes).view(np.uint8))
    return c.view(dt).to(torch.float64).numpy()


TIE_RTOL = 2.0 ** -18


def assert_codes_differ_only_at_ties(name: str, got, exp, q, fmt: str, rtol=TIE_RTOL):
    """Codes may differ by one FP8 step, and only where the oracle's quotient
    y / s (q, same shape) lies within rtol (relative) of the midpoint between
    the two codes' values: there a few ulp of exp error on the CUDA side decide
    the rounding direction.  Elsewhere the codes must be equal.  The clamped
    SwiGLU needs this form: clamping makes many y / s land exactly on an FP8
    midpoint (both factors of the ratio silu(c) / silu(c) cancel), so the
    differences there are not rare and independent."""
    got = np.ascontiguousarray(got)
    exp = np.ascontiguousarray(exp)
    d = np.abs(code_ordinal(got) - code_ordinal(exp))
    assert d.max(initial=0) <= 1, f"{name}: a code differs by {int(d.max())} steps"
    idx = np.nonzero(d)
    if idx[0].size == 0:
        return 0
    mid = (fp8_values(got[idx], fmt) + fp8_values(exp[idx], fmt)) / 2.0
    qq = np.asarray(q, np.float64)[idx]
    far = np.abs(qq - mid) > rtol * np.abs(mid)
    assert not far.any(), (f"{name}: {int(far.sum())} of {idx[0].size} differing codes are not "
                           f"at an FP8 tie; first quotient {qq[far][:4]} midpoint {mid[far][:4]}")
    return int(idx[0].size)
