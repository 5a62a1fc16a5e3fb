"""Host-side checks of the Python binding: caller-supplied output buffers are
refused, before anything is launched, when they are smaller than what the call
writes, not contiguous, on another device or of the wrong element size."""
from __future__ import annotations

import pytest
import torch

import fp8_activation_quantization_gb300 as tkq


def test_sf_shapes_match_the_c_byte_counts():
    # the binding's layout shapes against the library's own byte counts
    from fp8_activation_quantization_gb300 import _build
    _build.build()
    lib = tkq.load_library()
    for T in (0, 1, 5, 128, 1000, 8192):
        for G in (0, 1, 3, 4, 32, 57):
            for flags in (0, tkq.SF_ROUND_POW2, tkq.SF_COL_MAJOR,
                          tkq.SF_ROUND_POW2 | tkq.SF_UE8M0_PACKED,
                          tkq.SF_ROUND_POW2 | tkq.SF_UE8M0_PACKED | tkq.SF_COL_MAJOR):
                shape, dt = tkq._sf_shape(T, G, flags)
                assert 4 * shape[0] * shape[1] == lib.tkq_sf_bytes(T, G, flags), (T, G, flags)
                assert dt == ("int32" if flags & tkq.SF_UE8M0_PACKED else "float32")


def test_output_of_the_exact_size_is_accepted():
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    tkq._check_out(torch.empty(4 * 256, dtype=torch.uint8), "out", x, 4 * 256, itemsize=1)
    tkq._check_out(torch.empty(4, 256, dtype=torch.float8_e4m3fn), "out", x, 4 * 256, itemsize=1)
    tkq._check_sf_out(torch.empty(4, 2), "out_sf", x, 4, 2, 0)
    # a packed column-major layout, given as raw bytes
    tkq._check_sf_out(torch.empty(4 * 1 * 4, dtype=torch.uint8), "out_sf", x, 4, 2,
                      tkq.SF_ROUND_POW2 | tkq.SF_UE8M0_PACKED | tkq.SF_COL_MAJOR)


@pytest.mark.parametrize("bad, err", [
    (lambda: torch.empty(4 * 256 - 1, dtype=torch.uint8), ValueError),      # one byte short
    (lambda: torch.empty(256, 8, dtype=torch.uint8).t(), TypeError),         # not contiguous
    (lambda: torch.empty(4 * 256, dtype=torch.bfloat16), TypeError),         # 2-byte elements
    (lambda: None, TypeError),
])
def test_bad_code_buffers_are_refused(bad, err):
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(err):
        tkq._check_out(bad(), "out", x, 4 * 256, itemsize=1)


def test_short_scale_buffers_are_refused():
    x = torch.zeros(5, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        tkq._check_sf_out(torch.empty(5, 1), "out_sf", x, 5, 2, 0)
    # column-major pads the token count to a multiple of 4: [2, 8] floats, not [2, 5]
    with pytest.raises(ValueError):
        tkq._check_sf_out(torch.empty(2, 5), "out_sf", x, 5, 2, tkq.SF_COL_MAJOR)
    tkq._check_sf_out(torch.empty(2, 8), "out_sf", x, 5, 2, tkq.SF_COL_MAJOR)


def test_cast_back_output_type_is_pinned():
    x = torch.zeros(4, 128, dtype=torch.uint8)
    with pytest.raises(TypeError):
        tkq._check_out(torch.empty(4, 128, dtype=torch.float32), "out", x, 4 * 128 * 2,
                       dtype=torch.bfloat16)
