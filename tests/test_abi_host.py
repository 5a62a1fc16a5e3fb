"""Host-side checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every function declared in
include/tkq.h, and rejects invalid arguments with the documented status codes
before touching CUDA (no kernel is launched on these paths).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tkq.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_activation_quantization_gb300 import _build
    import fp8_activation_quantization_gb300 as tkq
    _build.build()
    return tkq.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*[\s\*]+(tkq_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tkq_per_token_cast", "tkq_swiglu_cast", "tkq_swiglu_cast_t", "tkq_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libtkq.so does not export {name}"


def test_checked_build_exports_every_declared_symbol(lib):
    """The access-checked test build compiles from the same sources, exports the
    same ABI and says which build it is; the release build says it is not."""
    from fp8_activation_quantization_gb300 import _build
    path = _build.build(checked=True)
    checked = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(checked, name), f"libtkq_checked.so does not export {name}"
    assert checked.tkq_checked_build() == 1
    assert lib.tkq_checked_build() == 0
    assert lib.tkq_read_check_address(None, 0) == 1           # NULL out-pointer


def test_library_is_built_for_sm_103a():
    from fp8_activation_quantization_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)
    assert os.path.exists(_build.LIB)


def test_status_strings(lib):
    import fp8_activation_quantization_gb300 as tkq
    for code, word in [(0, "TKQ_OK"), (1, "NULL"), (2, "SHAPE"), (3, "GROUP"), (4, "FMT"),
                       (5, "ALIGN"), (6, "CUDA"), (7, "TIMEOUT"), (8, "ALIAS"), (9, "FLAGS"),
                       (10, "VALUE"), (99, "UNKNOWN")]:
        assert word in tkq.tkq_status_string(code)


FAKE = 0x7F0000000000  # never dereferenced: every case below fails validation first
# the status codes of tkq.h that follow TKQ_ERR_CUDA = 6 and TKQ_ERR_TIMEOUT = 7
ALIAS, FLAGS, VALUE = 8, 9, 10


def p(off=0):
    return ctypes.c_void_p(FAKE + off)


@pytest.mark.parametrize("args,expected", [
    ((None, p(1 << 20), p(2 << 20), 4, 256, 128, 0), 1),          # NULL input
    ((p(), p(1 << 20), p(2 << 20), 4, 200, 128, 0), 2),           # C % 128
    ((p(), p(1 << 20), p(2 << 20), -1, 256, 128, 0), 2),          # T < 0
    ((p(), p(1 << 20), p(2 << 20), 4, 0, 128, 0), 2),             # C == 0
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 64, 0), 3),            # group
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 128, 2), 4),           # fmt
    ((p(8), p(1 << 20), p(2 << 20), 4, 256, 128, 0), 5),          # x misaligned
    ((p(), p((1 << 20) + 4), p(2 << 20), 4, 256, 128, 0), 5),     # out misaligned
    ((p(), p(1 << 20), p((2 << 20) + 2), 4, 256, 128, 0), 5),     # sf misaligned
    ((p(), p(512), p(2 << 20), 4, 256, 128, 0), ALIAS),               # out overlaps x
    ((p(), p(1 << 20), p((1 << 20) + 512), 4, 256, 128, 0), ALIAS),   # sf overlaps out
    ((None, None, None, 0, 256, 128, 0), 0),                      # empty batch
])
def test_per_token_cast_validation(lib, args, expected):
    assert lib.tkq_per_token_cast(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((p(), None, p(1 << 24), None, 4, 256, 128, 0), 1),
    ((p(), p((1 << 24) + 4), p(1 << 24), p(2 << 24), 4, 256, 128, 0), ALIAS),  # w overlaps out
    ((p(), p(4), p(1 << 24), p(2 << 24), 0, 256, 128, 0), 0),     # empty batch
    ((p(), p(1 << 26), p(1 << 24), p(2 << 24), 4, 100, 128, 0), 2),
    ((p(), p((1 << 26) + 2), p(1 << 24), p(2 << 24), 4, 256, 128, 0), 5),
    ((p(), None, p(1 << 24), p(2 << 24), 4, 256, 128, 3), 4),
])
def test_swiglu_cast_validation(lib, args, expected):
    assert lib.tkq_swiglu_cast(*args, None) == expected


@pytest.mark.parametrize("T,expected", [(100, 2), (0, 0), (-128, 2)])
def test_swiglu_cast_t_validation(lib, T, expected):
    if T == 0:
        args = (None, None, None, None, None, None, 0, 256, 128, 0, None)
    else:
        args = (p(), None, p(1 << 24), p(2 << 24), p(3 << 24), p(4 << 24), T, 256, 128, 0, None)
    assert lib.tkq_swiglu_cast_t(*args) == expected


@pytest.mark.parametrize("args,expected", [
    ((p(), None, None, p(1 << 24), p(2 << 24), 4, 256, 128, 0), 1),          # dy NULL
    ((p(), p(1 << 22), None, p(1 << 24), p(2 << 24), 4, 200, 128, 0), 2),    # H % 128
    ((p(), p((1 << 22) + 8), None, p(1 << 24), p(2 << 24), 4, 256, 128, 0), 5),  # dy misaligned
    ((p(), p(1 << 22), None, p(512), p(2 << 24), 4, 256, 128, 0), ALIAS),        # out overlaps x
    ((p(), p(1 << 22), None, p(1 << 24), p((1 << 24) + 64), 4, 256, 128, 0), ALIAS),  # sf in out
    ((None, None, None, None, None, 0, 256, 128, 0), 0),                       # empty batch
])
def test_swiglu_backward_validation(lib, args, expected):
    assert lib.tkq_swiglu_backward_cast(*args, None) == expected


def test_sf_bytes(lib):
    # T = 13 rows (T4 = 16), G = 7 groups (W = 2 words)
    assert lib.tkq_sf_bytes(13, 7, 0) == 13 * 7 * 4
    assert lib.tkq_sf_bytes(13, 7, 4) == 7 * 16 * 4
    assert lib.tkq_sf_bytes(13, 7, 2) == 13 * 2 * 4
    assert lib.tkq_sf_bytes(13, 7, 6) == 2 * 16 * 4
    assert lib.tkq_sf_bytes(13, 7, 1) == 13 * 7 * 4
    # the reciprocal reading leaves the layout alone
    assert lib.tkq_sf_bytes(13, 7, 8) == 13 * 7 * 4 and lib.tkq_sf_bytes(13, 7, 14) == 2 * 16 * 4
    assert lib.tkq_sf_bytes(13, 7, 16) == -1 and lib.tkq_sf_bytes(-1, 7, 0) == -1


@pytest.mark.parametrize("flags,sf_off,expected", [
    (16, 0, FLAGS),           # unknown flag bit
    (4, 4, 5),            # column-major scales must be 16-byte aligned
    (6, 8, 5),            # packed column-major too
    (2, 2, 5),            # packed row-major: 4-byte aligned
])
def test_ex_validation(lib, flags, sf_off, expected):
    args = (p(), p(1 << 24), p((2 << 24) + sf_off), 4, 256, 128, 0, flags, None)
    assert lib.tkq_per_token_cast_ex(*args) == expected


def test_ex_empty_batch_and_flags(lib):
    assert lib.tkq_per_token_cast_ex(None, None, None, 0, 256, 128, 0, 6, None) == 0
    assert lib.tkq_per_token_cast_ex(None, None, None, 0, 256, 128, 0, 9, None) == 0
    assert lib.tkq_per_token_cast_ex(None, None, None, 0, 256, 128, 0, 17, None) == FLAGS
    assert lib.tkq_swiglu_cast_ex(None, None, None, None, 0, 256, 128, 0, 16, None) == FLAGS
    assert lib.tkq_swiglu_backward_cast_ex(None, None, None, None, None, 0, 256, 128, 0, 4,
                                           None) == 0


def test_status_calls_validate_before_cuda(lib):
    assert lib.tkq_read_device_status(None, 0) == 1          # NULL flags
    assert lib.tkq_selftest_wait_timeout(0, None) == 2       # limit out of range
    assert lib.tkq_selftest_wait_timeout(3_000_000_000, None) == 2


def test_swiglu_cast_t_output_alias(lib):
    # out_t overlapping out
    assert lib.tkq_swiglu_cast_t(p(), None, p(1 << 24), p(2 << 24), p((1 << 24) + 256),
                                 p(4 << 24), 128, 256, 128, 0, None) == ALIAS


@pytest.mark.parametrize("args,expected", [
    ((None, p(1 << 20), p(2 << 20), 256, 256, 128, 0, 0), 1),         # NULL input
    ((p(), p(1 << 20), p(2 << 20), 200, 256, 128, 0, 0), 2),          # T % 128
    ((p(), p(1 << 20), p(2 << 20), 256, 200, 128, 0, 1), 2),          # C % 128
    ((p(), p(1 << 20), p(2 << 20), 256, 256, 32, 0, 0), 3),           # group
    ((p(), p(1 << 20), p(2 << 20), 256, 256, 128, 5, 0), 4),          # fmt
    ((p(), p((1 << 20) + 8), p(2 << 20), 256, 256, 128, 0, 1), 5),    # out misaligned
    ((p(), p(1 << 20), p((2 << 20) + 1), 256, 256, 128, 0, 0), 5),    # sf misaligned
    ((p(), p(1 << 16), p(2 << 20), 256, 256, 128, 0, 0), ALIAS),          # out overlaps x
    ((p(), p(1 << 20), p((1 << 20) + 4096), 256, 256, 128, 0, 1), ALIAS), # sf overlaps out
    ((None, None, None, 0, 256, 128, 0, 1), 0),                       # empty batch
])
def test_per_channel_cast_validation(lib, args, expected):
    assert lib.tkq_per_channel_cast(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((p(), None, p(2 << 20), 300, 256, 128, 0), 1),                   # NULL out
    ((p(), p(1 << 20), p(2 << 20), 300, 200, 128, 0), 2),             # C % 128
    ((p(), p(1 << 20), p(2 << 20), 300, 256, 256, 0), 3),             # block
    ((p(), p(1 << 20), p(2 << 20), 300, 256, 128, -1), 4),            # fmt
    ((p(4), p(1 << 20), p(2 << 20), 300, 256, 128, 0), 5),            # x misaligned
    ((p(), p(1 << 20), p((1 << 20) + 65536), 300, 256, 128, 0), ALIAS),   # sf overlaps out
    ((None, None, None, 0, 256, 128, 0), 0),                          # empty batch
])
def test_per_block_cast_validation(lib, args, expected):
    assert lib.tkq_per_block_cast(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((None, p(1 << 20), p(2 << 20), 4, 256, 1, 128, 0, 0), 1),        # NULL codes
    ((p(), p(1 << 20), p(2 << 20), 4, 200, 1, 128, 0, 0), 2),         # C % 128
    ((p(), p(1 << 20), p(2 << 20), -2, 256, 1, 128, 0, 0), 2),        # T < 0
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 1, 1, 0, 0), 3),           # 1 x 1 groups
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 128, 64, 0, 0), 3),        # 128 x 64 groups
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 1, 128, 3, 0), 4),         # fmt
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 1, 128, 0, 2), 4),         # out dtype
    ((p(), p((1 << 20) + 4), p(2 << 20), 4, 256, 128, 1, 0, 0), 5),   # per-channel sf / 16
    ((p(), p(1 << 20), p((2 << 20) + 8), 4, 256, 1, 128, 0, 1), 5),   # out misaligned
    ((p(), p(1 << 20), p(512), 4, 256, 1, 128, 0, 0), ALIAS),             # out overlaps codes
    ((p(), p(1 << 20), p((1 << 20) - 1024), 4, 256, 1, 128, 0, 1), ALIAS),  # out overlaps sf
    ((None, None, None, 0, 256, 128, 128, 1, 1), 0),                  # empty batch
])
def test_cast_back_validation(lib, args, expected):
    assert lib.tkq_cast_back(*args, None) == expected


@pytest.mark.parametrize("clamp,count_off,expected", [
    (0.0, 0, VALUE),              # bound must be > 0
    (-1.0, 0, VALUE),
    (float("inf"), 0, VALUE),
    (float("nan"), 0, VALUE),
    (4.0, 4, 5),              # counter not 8-byte aligned
    (4.0, -(4 << 20) + 64, ALIAS),   # counter inside x
    (4.0, -(1 << 20) + 64, ALIAS),   # counter inside out
])
def test_swiglu_clamp_validation(lib, clamp, count_off, expected):
    T, H = 256, 256
    count = p((4 << 20) + count_off)
    args = (p(), None, p(3 << 20), p(5 << 20), T, H, 128, 0, 0, clamp, count, None)
    assert lib.tkq_swiglu_cast_clamp(*args) == expected
    args_t = (p(), None, p(3 << 20), p(5 << 20), p(6 << 20), p(7 << 20), T, H, 128, 0, 0, clamp,
              count, None)
    assert lib.tkq_swiglu_cast_t_clamp(*args_t) == expected


def test_swiglu_clamp_empty_batch_checks_the_bound(lib):
    assert lib.tkq_swiglu_cast_clamp(None, None, None, None, 0, 256, 128, 0, 0, 1.0, None, None) == 0
    assert lib.tkq_swiglu_cast_clamp(None, None, None, None, 0, 256, 128, 0, 0, 0.0, None, None) == VALUE
    assert "VALUE" in __import__("fp8_activation_quantization_gb300").tkq_status_string(VALUE)


@pytest.mark.parametrize("args,expected", [
    ((None, p(1 << 20), p(2 << 20), 4, 256, 128, 0, 0), 1),            # NULL input
    ((p(), p(1 << 20), p(2 << 20), 4, 200, 128, 0, 0), 2),             # C % 128
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 64, 0, 0), 3),              # group
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 128, 7, 0), 4),             # fmt
    ((p(), p(1 << 20), p(2 << 20), 4, 256, 128, 0, 16), FLAGS),            # flags
    ((p(4), p(1 << 20), p(2 << 20), 4, 256, 128, 0, 0), 5),            # x misaligned
    ((p(), p(2048), p(2 << 20), 4, 256, 128, 0, 0), ALIAS),                # out inside x (4 B/elem)
    ((None, None, None, 0, 256, 128, 0, 0), 0),                        # empty batch
])
def test_per_token_cast_f32_validation(lib, args, expected):
    assert lib.tkq_per_token_cast_f32(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((None, None, p(1 << 24), 4, 128), 1),                 # NULL x
    ((p(), None, p(1 << 24), 4, 100), 2),                  # H % 128
    ((p(4), None, p(1 << 24), 4, 128), 5),                 # x misaligned
    ((p(), p(2), p(1 << 24), 4, 128), 5),                  # w misaligned
    ((p(), None, p(1024), 4, 128), ALIAS),                     # y inside x (2048 bytes)
    ((None, None, None, 0, 128), 0),                       # empty batch
])
def test_swiglu_values_validation(lib, args, expected):
    assert lib.tkq_swiglu_values(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((p(), None, None, p(1 << 24), 4, 128), 1),             # NULL dy
    ((p(), p(1 << 20), None, p(1 << 24), 4, 200), 2),       # H % 128
    ((p(), p((1 << 20) + 8), None, p(1 << 24), 4, 128), 5),  # dy misaligned
    ((p(), p(1 << 20), None, p((1 << 24) + 4), 4, 128), 5),  # y misaligned
    ((p(), p(1 << 20), None, p((1 << 20) + 512), 4, 128), ALIAS),  # y overlaps dy (1024 bytes)
    ((p(), p(1 << 20), p(1 << 22), p((1 << 22) - 4096 + 16), 4, 128), ALIAS),  # w inside y
    ((None, None, None, None, 0, 128), 0),                  # empty batch
])
def test_swiglu_backward_values_validation(lib, args, expected):
    assert lib.tkq_swiglu_backward_values(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((p(), p(1 << 24), 6, 0), 2),             # n % 4
    ((p(), p(1 << 24), -4, 0), 2),            # n < 0
    ((p(), p(1 << 24), 16, 3), 4),            # fmt
    ((None, p(1 << 24), 16, 0), 1),           # NULL x
    ((p(8), p(1 << 24), 16, 0), 5),           # x misaligned
    ((p(), p(2), 16, 0), 5),                  # out misaligned
    ((p(), p(32), 16, 0), ALIAS),                 # out inside x (64 bytes)
    ((None, None, 0, 1), 0),                  # empty
])
def test_fp8_encode_validation(lib, args, expected):
    assert lib.tkq_fp8_encode(*args, None) == expected


@pytest.mark.parametrize("flags,sf_t_addr,expected", [
    (16, 7 << 20, FLAGS),                      # unknown flag bit
    (4, (7 << 20) + 4, 5),                 # column-major sf_t must be 16-byte aligned
    (0, (7 << 20) + 4, 0),                 # empty batch: valid flags return OK, no launch
    (6, (5 << 20) + 16, ALIAS),                # sf_t inside sf (both sized by their layouts)
])
def test_swiglu_cast_t_ex_validation(lib, flags, sf_t_addr, expected):
    T, H = (0 if expected == 0 else 256), 256
    args = (p(), None, p(3 << 20), p(5 << 20), p(6 << 20), p(sf_t_addr), T, H, 128, 0, flags,
            None)
    assert lib.tkq_swiglu_cast_t_ex(*args) == expected
