"""The oracle's FP8 encoder on every one of the 2^32 binary32 bit patterns,
against two references:
1. torch's float8 conversion (a library routine, round to nearest even) with
   the saturation rule applied on top: where torch gives a finite code the
   oracle gives the same; where a finite input overflows (torch: NaN for
   e4m3fn, inf for e5m2) the oracle gives the largest finite code of that
   sign; an infinite input gives the largest finite code of its sign; a NaN
   gives the NaN code 0x7F (either sign bit accepted);
2. a brute-force nearest-value search: the finite codes of each format are
   decoded by torch (their magnitudes increase with the code), and |v| is
   placed among the midpoints between consecutive magnitudes; the nearer
   magnitude wins, an exact midpoint goes to the even code (even last mantissa
   bit), anything above the largest finite magnitude saturates to it, and the
   sign bit is copied.
Split over threads (ctypes, torch and numpy release the GIL); every thread
reuses its buffers."""
import os
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

CHUNK = 1 << 22
MAXCODE = {"e4m3": 0x7E, "e5m2": 0x7B}
TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
_BASE = np.arange(CHUNK, dtype=np.uint32)
_local = threading.local()


def _magnitudes(fmt):
    """Decoded magnitudes of the non-negative finite codes 0 .. MAXCODE."""
    codes = torch.arange(MAXCODE[fmt] + 1, dtype=torch.uint8)
    return codes.view(TORCH[fmt]).to(torch.float64).numpy()


MAGS = {f: _magnitudes(f) for f in MAXCODE}


def _midpoints(fmt):
    """Binary32 bit patterns of the midpoints between consecutive magnitudes
    (every such midpoint is exactly a binary32 value)."""
    m = MAGS[fmt]
    mid = (m[:-1] + m[1:]) / 2.0
    assert np.array_equal(mid.astype(np.float32).astype(np.float64), mid)
    return mid.astype(np.float32).view(np.uint32)


MIDS = {f: _midpoints(f) for f in MAXCODE}


def _nearest_codes(bits, fmt):
    """The brute-force encoder (reference 2) for non-NaN bit patterns.  Positive
    binary32 patterns order like their values, so the number of midpoints below
    |v| is the index of the nearest magnitude; |v| equal to a midpoint is a tie
    between codes k and k + 1, which goes to the even one; beyond the largest
    magnitude every midpoint is below, which saturates."""
    mids = MIDS[fmt]
    mag = bits & np.uint32(0x7FFFFFFF)
    k = np.searchsorted(mids, mag).astype(np.uint8)          # at most MAXCODE
    tie = mids[np.minimum(k, np.uint8(mids.size - 1))] == mag
    code = k + (tie & ((k & np.uint8(1)) == 1)).astype(np.uint8)
    return code | ((bits >> np.uint32(24)).astype(np.uint8) & np.uint8(0x80))


def _buffers(fmt):
    b = getattr(_local, fmt, None)
    if b is None:
        b = {"bits": np.empty(CHUNK, np.uint32), "got": np.empty(CHUNK, np.uint8),
             "ref": torch.empty(CHUNK, dtype=TORCH[fmt]), "val": torch.empty(CHUNK)}
        setattr(_local, fmt, b)
    return b


def _check_chunk(start, fmt):
    b = _buffers(fmt)
    bits = b["bits"]
    np.add(_BASE, np.uint32(start), out=bits)
    v = bits.view(np.float32)
    got = oracle.fp8_encode_array(v, fmt, out=b["got"])
    b["ref"].copy_(torch.from_numpy(v))
    b["val"].copy_(b["ref"])
    ref = b["ref"].view(torch.uint8).numpy()
    nan_in = np.isnan(v)
    overflow = ~nan_in & ~np.isfinite(b["val"].numpy())   # torch: NaN or inf for a non-NaN input
    sat = ((bits >> np.uint32(24)).astype(np.uint8) & np.uint8(0x80)) | np.uint8(MAXCODE[fmt])
    exp = np.where(overflow, sat, ref)
    bad = np.where(nan_in, (got & np.uint8(0x7F)) != np.uint8(0x7F), got != exp)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        return f"{fmt}: bits {int(bits[i]):#010x} -> {int(got[i]):#04x}, expected {int(exp[i]):#04x}"
    near = _nearest_codes(bits, fmt)
    bad = ~nan_in & (got != near)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        return (f"{fmt}: bits {int(bits[i]):#010x} -> {int(got[i]):#04x}, nearest-value search "
                f"{int(near[i]):#04x}")
    return None


@pytest.mark.slow
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encoder_on_all_2_32_bit_patterns(fmt):
    workers = max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        errs = [e for e in ex.map(lambda s: _check_chunk(s, fmt), range(0, 1 << 32, CHUNK)) if e]
    assert not errs, errs[:4]
