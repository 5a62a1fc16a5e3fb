"""The hardware FP8 conversion (cvt.rn.satfinite, the last step of every cast)
on every one of the 2^32 binary32 bit patterns, through tkq_fp8_encode,
against the oracle's encoder: bit-identical codes for every non-NaN input
(finite values of any magnitude, saturation beyond the largest finite value,
infinities to the largest finite code of their sign, signed zeros, every
subnormal), and a NaN code of the format for every NaN input (the oracle gives
0x7F; the hardware's choice of NaN pattern and sign is accepted).  The casts
alone never hand the conversion values beyond about fmt_max, so this is the
check of the saturation and NaN semantics."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CHUNK = 1 << 28            # values per launch (divides 2^31: no chunk crosses the sign bit)
SUB = 1 << 22              # values per oracle call
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def _is_nan_code(c, fmt):
    if fmt == "e4m3":
        return (c & 0x7F) == 0x7F
    return ((c & 0x7C) == 0x7C) & ((c & 0x03) != 0)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_conversion_on_every_bit_pattern(cuda_device, fmt):
    dev = cuda_device
    exp = np.empty(CHUNK, np.uint8)
    errors = []
    with ThreadPoolExecutor(THREADS) as ex:
        for start in range(0, 1 << 32, CHUNK):
            first = start if start < (1 << 31) else start - (1 << 32)   # as a signed int32
            xd = torch.arange(first, first + CHUNK, dtype=torch.int32, device=dev).view(torch.float32)
            got = tkq.fp8_encode(xd, fmt).cpu().numpy()
            del xd
            bits = np.arange(start, start + CHUNK, dtype=np.uint32)
            v = bits.view(np.float32)
            list(ex.map(lambda a: oracle.fp8_encode_array(v[a:a + SUB], fmt, out=exp[a:a + SUB]),
                        range(0, CHUNK, SUB)))
            nan = np.isnan(v)
            bad = np.where(nan, ~_is_nan_code(got, fmt), got != exp)
            if bad.any():
                i = int(np.flatnonzero(bad)[0])
                errors.append(f"bits {int(bits[i]):#010x}: hardware {int(got[i]):#04x}, "
                              f"oracle {int(exp[i]):#04x} ({int(bad.sum())} in this chunk)")
    assert not errors, errors[:4]
    assert tkq.tkq_read_device_status() == 0
