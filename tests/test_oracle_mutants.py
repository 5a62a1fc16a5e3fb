"""The oracle's pins must reject plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a wrong
constant, a wrong rounding tie rule, a dropped term, a swapped operand, a
transposed index ...), builds that copy on the CPU, routes the oracle module
to it, and requires that at least one pin of tests/test_oracle_pins.py fails.
The real oracle is never modified.
"""
import os

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tkq_oracle.c")

MUTANTS = [
    ("clamp minimum 1e-3", "const float clamp_min = 1e-4f;", "const float clamp_min = 1e-3f;"),
    ("ties to odd", "fmod(r, 2.0) != 0.0", "fmod(r, 2.0) == 0.0"),
    ("ties away from zero", "frac > 0.5 ||", "frac >= 0.5 ||"),
    ("saturate to NaN", "return (uint8_t)(sign | d.maxcode);   /* satfinite */",
     "return (uint8_t)(sign | 0x7F);"),
    ("quotient by reciprocal multiply", "const float q = v[i * stride] / s;",
     "const float q = v[i * stride] * (1.0f / s);"),
    ("no subnormal quantum", "if (e < emin) e = emin;", ""),
    ("sign of zero lost", "const uint8_t sign = signbit(v) ? 0x80 : 0x00;",
     "const uint8_t sign = (v < 0) ? 0x80 : 0x00;"),
    ("last value instead of max", "if (a > amax) amax = a;", "amax = a;"),
    ("gate and up swapped", "const float silu = g / den;\n            float val = silu * u;",
     "const float silu = u / (1.0f + (float)exp(-(double)u));\n            float val = silu * g;"),
    ("exp sign flipped", "exp(-(double)g)", "exp((double)g)"),
    ("1 - exp", "const float den = 1.0f + e;", "const float den = 1.0f - e;"),
    ("routing weight dropped", "if (w) val = val * w[t];", ""),
    ("token-axis operand transposed", "y + (b * group) * C + c, group, C,",
     "y + c * T + b * group, group, 1,"),
    ("E4M3 bias 8", "d->mbits = 3; d->ebits = 4; d->bias = 7;",
     "d->mbits = 3; d->ebits = 4; d->bias = 8;"),
    ("E4M3 max code 0x7D", "d->maxval = 448.0; d->maxcode = 0x7E;",
     "d->maxval = 448.0; d->maxcode = 0x7D;"),
    ("E5M2 max 61440", "d->maxval = 57344.0; d->maxcode = 0x7B;",
     "d->maxval = 61440.0; d->maxcode = 0x7B;"),
    ("scale from the first element", "const float s = ora_group_scale(amax, fmt);",
     "const float s = ora_group_scale(fabsf(v[0]), fmt);"),
    ("backward: 1 + sigma in dsilu", "const double dsilu = sig * (1.0 + g * (1.0 - sig));",
     "const double dsilu = sig * (1.0 + g * (1.0 + sig));"),
    ("backward: dg and du swapped", "grad[t * 2 * H + c] = (float)(d * u * dsilu * wt);",
     "grad[t * 2 * H + H + c] = (float)(d * u * dsilu * wt); continue;"),
    ("backward: weight dropped from du", "grad[t * 2 * H + H + c] = (float)(d * silu * wt);",
     "grad[t * 2 * H + H + c] = (float)(d * silu);"),
    ("scale rounded down to a power of two", "return (float)ldexp(1.0, e);",
     "return (float)ldexp(1.0, e - 1);"),
    ("UE8M0 bytes in reverse order", "((uint8_t*)sf)[word * 4 + j % 4]",
     "((uint8_t*)sf)[word * 4 + 3 - j % 4]"),
    ("column-major scales without padding", "((float*)sf)[cm ? j * T4 + t : t * G + j] = s;",
     "((float*)sf)[cm ? j * T + t : t * G + j] = s;"),
    ("per-channel codes written along the row",
     "sf[b * C + c] = cast_group(v, group, 1, fmt, out + (b * group) * C + c, C);",
     "sf[b * C + c] = cast_group(v, group, 1, fmt, out + (b * group) * C + c, 1);"),
    ("per-block scale from the first row only",
     "const float s = ora_group_scale(group_absmax(v, rows * block, 1), fmt);",
     "const float s = ora_group_scale(group_absmax(v, block, 1), fmt);"),
    ("clamp: gate clamped from below too", "if (g > cv) { g = cv; ++n; }",
     "if (g > cv) { g = cv; ++n; }\n                if (g < -cv) { g = -cv; ++n; }"),
    ("clamp: up clamped from above only", "if (u < -cv) { u = -cv; ++n; }", ""),
    ("clamp: clamped ups not counted", "if (u > cv) { u = cv; ++n; }", "if (u > cv) { u = cv; }"),
    ("clamp: values at the bound counted", "if (g > cv) { g = cv; ++n; }",
     "if (g >= cv) { g = cv; ++n; }"),
    ("reciprocal reading ignored", "            if (reciprocal)\n", "            if (0)\n"),
    ("reciprocal reading multiplies by s", "const float q = v[i] * inv;",
     "const float q = v[i] * s;"),
    ("cast back ignores the column group", "const float s = sf[(t / gr) * G + c / gc];",
     "const float s = sf[(t / gr) * G];"),
]

# cheapest first: most mistakes are caught by the hand-worked fixtures
CHECKS = [
    (pins.test_hand_groups, {}),
    (pins.test_encode_hand_points, {}),
    (pins.test_decode_hand_points, {}),
    (pins.test_zero_row_and_signed_zero, {}),
    (pins.test_swiglu_orientation_and_special_cases, {}),
    (pins.test_swiglu_weight_one_and_weight_product, {}),
    (pins.test_swiglu_vs_binary64, {}),
    (pins.test_swiglu_backward_special_cases, {}),
    (pins.test_round_pow2_hand_group, {}),
    (pins.test_reciprocal_reading_hand_groups, {}),
    (pins.test_swiglu_clamp_hand_values, {}),
    (pins.test_cast_back_hand_values_and_granularities, {}),
    (pins.test_per_channel_is_per_token_of_transpose, {"fmt": "e4m3"}),
    (pins.test_per_block_is_per_token_of_flattened_blocks, {"fmt": "e4m3", "T": 300}),
    (pins.test_pow2_ceil_against_numpy_and_properties, {}),
    (pins.test_sf_layouts_rearrange_the_row_major_scales, {"flags": oracle.SF_COL_MAJOR}),
    (pins.test_sf_layouts_rearrange_the_row_major_scales,
     {"flags": oracle.SF_UE8M0_PACKED | oracle.SF_COL_MAJOR}),
    (pins.test_swiglu_backward_vs_finite_differences, {}),
    (pins.test_cols_equal_rows_of_transpose, {"fmt": "e4m3"}),
    (pins.test_cols_index_orientation, {}),
    (pins.test_scale_floor_amax_code_and_error_bound, {"fmt": "e4m3"}),
    (pins.test_scale_floor_amax_code_and_error_bound, {"fmt": "e5m2"}),
    (pins.test_negation_flips_only_sign, {"fmt": "e4m3"}),
    (pins.test_permutation_within_group, {"fmt": "e4m3"}),
    (pins.test_decode_all_codes_match_torch, {"fmt": "e4m3"}),
    (pins.test_decode_all_codes_match_torch, {"fmt": "e5m2"}),
    (pins.test_encode_matches_brute_force, {"fmt": "e4m3"}),
    (pins.test_encode_matches_brute_force, {"fmt": "e5m2"}),
]


def test_pins_pass_on_the_real_oracle():
    for fn, kw in CHECKS:
        fn(**kw)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not found exactly once"
    lib = oracle.build_variant(src.replace(old, new), str(tmp_path))
    caught = None
    with oracle.use_library(lib):
        for fn, kw in CHECKS:
            try:
                fn(**kw)
            except Exception as e:  # AssertionError, ValueError ...
                caught = f"{fn.__name__}{kw}: {type(e).__name__}"
                break
    assert caught is not None, f"no pin rejects the planted mistake {name!r}"
