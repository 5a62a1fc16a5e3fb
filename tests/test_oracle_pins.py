"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
* the FP8 decode of all 256 codes against torch's float8 dtypes (a library
  routine) and against hand-worked code values;
* the encoder against a brute-force nearest-value search over the 256 decoded
  values (a different algorithm from the oracle's bit rounding), against torch's
  round-to-nearest conversion in range, and against hand-worked points;
* the group cast against hand-worked 1x128 groups (tests/golden);
* invariants that hold for any input: sign symmetry, exact 2^k scale
  equivariance, permutation equivariance, the half-spacing error bound, the
  clamp floor, the amax element mapping to the largest code;
* SwiGLU against a binary64 evaluation and torch's silu, the gate/up
  orientation, w = 1 and zero-gate special cases;
* the token-axis cast against the channel-axis cast of the explicit transpose.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_activation_quantization_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
MAXCODE = {"e4m3": 0x7E, "e5m2": 0x7B}
FMAX = {"e4m3": 448.0, "e5m2": 57344.0}
MBITS = {"e4m3": 3, "e5m2": 2}
EMIN = {"e4m3": -6, "e5m2": -14}
FMTS = ["e4m3", "e5m2"]


def torch_decode_all(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def _val(spec):
    if isinstance(spec, dict):
        (k, v), = spec.items()
        f = np.float32(v)
        return np.nextafter(f, np.float32(np.inf if k == "nextup" else -np.inf), dtype=np.float32)
    if isinstance(spec, str):
        return np.float32(float(spec))
    return np.float32(spec)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_decode_all_codes_match_torch(fmt):
    ref = torch_decode_all(fmt)
    got = np.array([oracle.fp8_decode(c, fmt) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_hand_points():
    pts = json.load(open(os.path.join(GOLDEN, "codec_points.json")))["decode"]
    for fmt, code, val in pts:
        got = oracle.fp8_decode(int(code, 16), fmt)
        if val == "nan":
            assert math.isnan(got), (fmt, code)
        else:
            exp = float(val)
            assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (fmt, code, got)


def test_fp8_max():
    assert oracle.fp8_max("e4m3") == 448.0 and oracle.fp8_max("e5m2") == 57344.0


# ---------------------------------------------------------------------------
# encode
# ---------------------------------------------------------------------------

def brute_force_encode(v: np.ndarray, fmt: str) -> np.ndarray:
    """Nearest finite FP8 value by exhaustive search over the torch-decoded
    table; ties go to the code with an even mantissa (even code); magnitudes at
    or above the largest finite value saturate; NaN -> 0x7F; sign kept."""
    table = torch_decode_all(fmt)
    maxcode = MAXCODE[fmt]
    pos_codes = np.arange(0, maxcode + 1)
    pos_vals = table[pos_codes]
    assert np.all(np.diff(pos_vals) > 0)
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    out = np.zeros(v.shape, np.uint8)
    nan = np.isnan(v)
    a_f = np.where(nan, 0.0, a)
    # distance to every finite code (small tables: brute force is cheap)
    res = np.empty(v.shape, np.int64)
    B = 1 << 16
    flat_a = a_f.ravel()
    flat_res = res.ravel()
    for s in range(0, flat_a.size, B):
        d = np.abs(flat_a[s:s + B, None] - pos_vals[None, :])
        best = d.min(axis=1, keepdims=True)
        cand = d == best
        # among the nearest, prefer an even code
        even = cand & ((pos_codes[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        flat_res[s:s + B] = pos_codes[pick]
    res = flat_res.reshape(v.shape)
    res = np.where(a_f >= FMAX[fmt], maxcode, res)
    sign = np.signbit(v).astype(np.uint8) << 7
    out[...] = (res | sign).astype(np.uint8)
    out[nan] = 0x7F
    return out


def encode_test_points(fmt: str, n_random: int = 400_000, seed: int = 7) -> np.ndarray:
    table = torch_decode_all(fmt)
    pos = table[: MAXCODE[fmt] + 1].astype(np.float32)
    mids = ((table[: MAXCODE[fmt]] + table[1: MAXCODE[fmt] + 1]) / 2).astype(np.float32)
    extra = np.array([FMAX[fmt] * 1.03125, FMAX[fmt] * 1.0625, FMAX[fmt] * 1.07, FMAX[fmt] * 2,
                      1e30, np.inf, 1e-45, 1e-40, 1.17549435e-38, 0.0], np.float32)
    base = np.concatenate([pos, mids, extra])
    pts = [base]
    for k in (1, 2, 3):
        up = base.copy()
        dn = base.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf), dtype=np.float32)
            dn = np.nextafter(dn, np.float32(-np.inf), dtype=np.float32)
        pts += [up, dn]
    rng = np.random.default_rng(seed)
    e = rng.integers(EMIN[fmt] - 14, int(math.log2(FMAX[fmt])) + 3, n_random)
    m = rng.random(n_random) + 1.0
    pts.append((m * np.exp2(e)).astype(np.float32))
    bits = rng.integers(0, 2 ** 31 - 1, 50_000, dtype=np.int64).astype(np.uint32)
    rnd = bits.view(np.float32)
    pts.append(rnd[np.isfinite(rnd)])
    allp = np.concatenate(pts)
    allp = allp[~np.isnan(allp)]
    return np.concatenate([allp, -allp])


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_matches_brute_force(fmt):
    v = encode_test_points(fmt)
    got = oracle.fp8_encode_array(v, fmt)
    ref = brute_force_encode(v, fmt)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_matches_torch_in_range(fmt):
    v = encode_test_points(fmt, n_random=200_000, seed=11)
    v = v[np.abs(v) <= FMAX[fmt]]
    ref = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    got = oracle.fp8_encode_array(v, fmt)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_hand_points():
    pts = json.load(open(os.path.join(GOLDEN, "codec_points.json")))["encode"]
    for fmt, val, code in pts:
        v = _val(val)
        assert oracle.fp8_encode(v, fmt) == int(code, 16), (fmt, val, float(v))


@pytest.mark.parametrize("fmt", FMTS)
def test_encode_decode_roundtrip_all_codes(fmt):
    table = torch_decode_all(fmt)
    for c in range(256):
        if not np.isfinite(table[c]):
            continue
        assert oracle.fp8_encode(np.float32(table[c]), fmt) == c, hex(c)


# ---------------------------------------------------------------------------
# group cast: hand-worked groups
# ---------------------------------------------------------------------------

def _bf16_exact(vals: np.ndarray) -> np.ndarray:
    bits = synth.f32_to_bf16_bits(vals)
    assert np.array_equal(synth.bf16_bits_to_f32(bits).view(np.uint32),
                          vals.astype(np.float32).view(np.uint32)), "not bf16-exact"
    return bits


def test_hand_groups():
    spec = json.load(open(os.path.join(GOLDEN, "hand_groups.json")))
    G = spec["group"]
    for case in spec["cases"]:
        vals = np.full(G, case["fill"], np.float32)
        for k, v in case["set"].items():
            vals[int(k)] = np.float32(v)
        bits = _bf16_exact(vals).reshape(1, G)
        codes, sf = oracle.per_token_cast(bits, case["fmt"], G)
        assert sf.shape == (1, 1)
        assert hex(int(sf.view(np.uint32)[0, 0])) == case["scale_hex"], case["name"]
        exp = np.full(G, int(case["code_fill"], 16), np.uint8)
        for k, c in case["codes"].items():
            exp[int(k)] = int(c, 16)
        bad = np.nonzero(codes[0] != exp)[0]
        assert bad.size == 0, (case["name"], [(int(i), hex(codes[0, i]), hex(exp[i])) for i in bad])


# ---------------------------------------------------------------------------
# group cast: invariants on seeded random data
# ---------------------------------------------------------------------------

def _random_bits(T=96, C=1024, seed=3, outliers=True):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, C)).astype(np.float32)
    if outliers:
        m = rng.random((T, C)) < 0.002
        v[m] *= 300.0
    v[5] = 0.0
    v[6, :128] = np.float32(3e-5) * np.sign(v[6, :128])  # clamped group
    return synth.f32_to_bf16_bits(v)


@pytest.mark.parametrize("fmt", FMTS)
def test_negation_flips_only_sign(fmt):
    x = _random_bits()
    c1, s1 = oracle.per_token_cast(x, fmt)
    c2, s2 = oracle.per_token_cast(x ^ np.uint16(0x8000), fmt)
    assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    assert np.array_equal(c2, c1 ^ np.uint8(0x80))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("k", [-7, 3])
def test_power_of_two_scaling(fmt, k):
    x = _random_bits(outliers=False, seed=5)
    xf = synth.bf16_bits_to_f32(x)
    xf = np.where(np.abs(xf) < 2.0 ** -60, np.float32(0), xf)  # keep far from bf16 underflow
    x = synth.f32_to_bf16_bits(xf)
    keep = np.ones(x.shape[0], bool)
    keep[[5, 6]] = False  # zero / clamped rows change scale non-proportionally
    x = x[keep]
    xs = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
    assert np.array_equal(synth.bf16_bits_to_f32(xs), synth.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
    c1, s1 = oracle.per_token_cast(x, fmt)
    c2, s2 = oracle.per_token_cast(xs, fmt)
    assert np.array_equal(c1, c2)
    assert np.array_equal(s2, s1 * np.float32(2.0 ** k))


@pytest.mark.parametrize("fmt", FMTS)
def test_permutation_within_group(fmt):
    x = _random_bits(seed=9)
    T, C = x.shape
    perm = np.random.default_rng(1).permutation(128)
    xp = x.reshape(T, C // 128, 128)[:, :, perm].reshape(T, C)
    c1, s1 = oracle.per_token_cast(x, fmt)
    c2, s2 = oracle.per_token_cast(xp, fmt)
    assert np.array_equal(s1, s2)
    assert np.array_equal(c2, c1.reshape(T, C // 128, 128)[:, :, perm].reshape(T, C))


@pytest.mark.parametrize("fmt", FMTS)
def test_scale_floor_amax_code_and_error_bound(fmt):
    x = _random_bits(seed=13)
    codes, sf = oracle.per_token_cast(x, fmt)
    T, C = x.shape
    G = C // 128
    v = synth.bf16_bits_to_f32(x).astype(np.float64).reshape(T, G, 128)
    s = sf.astype(np.float64).reshape(T, G, 1)
    floor = np.float32(1e-4) / np.float32(FMAX[fmt])
    assert np.all(sf >= floor)
    amax = np.abs(v).max(axis=2)
    # scale is amax / fmt_max to within half a binary32 ulp where not clamped
    big = amax > 1e-4
    rel = np.abs(sf.astype(np.float64)[big] * FMAX[fmt] - amax[big]) / amax[big]
    assert rel.max() <= 2.0 ** -24 * 1.0001
    # the element attaining amax gets the largest code
    arg = np.abs(v).argmax(axis=2)
    c = codes.reshape(T, G, 128)
    top = np.take_along_axis(c, arg[..., None], axis=2)[..., 0]
    assert np.all((top & 0x7F)[big] == MAXCODE[fmt])
    # |dec(q) - v/s| <= half the FP8 spacing at v/s (+ the binary32 quotient rounding)
    table = torch_decode_all(fmt)
    dec = table[c]
    q = v / s
    e = np.floor(np.log2(np.maximum(np.abs(q), 1e-300)))
    e = np.maximum(e, EMIN[fmt])
    half = 0.5 * np.exp2(e - MBITS[fmt])
    err = np.abs(dec - q)
    assert np.all(err <= half * (1 + 2.0 ** -20) + np.abs(q) * 2.0 ** -23)


def test_zero_row_and_signed_zero():
    x = np.zeros((2, 256), np.uint16)
    x[1, 3] = 0x8000  # -0.0
    c, s = oracle.per_token_cast(x, "e4m3")
    assert np.all(s == np.float32(1e-4) / np.float32(448))
    assert c[1, 3] == 0x80 and np.count_nonzero(c) == 1


# ---------------------------------------------------------------------------
# token-axis cast
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_cols_equal_rows_of_transpose(fmt):
    rng = np.random.default_rng(21)
    y = rng.standard_normal((256, 384)).astype(np.float32) * np.float32(3)
    y[:128, 7] = 0.0
    y[128:, 9] *= np.float32(1e3)
    ct, st = oracle.cast_cols_f32(y, fmt)
    cr, sr = oracle.cast_rows_f32(np.ascontiguousarray(y.T), fmt)
    assert ct.shape == (384, 256) and st.shape == (384, 2)
    assert np.array_equal(ct, cr) and np.array_equal(st.view(np.uint32), sr.view(np.uint32))


def test_cols_index_orientation():
    # distinct column magnitudes: column c of the input is scaled by (c + 1),
    # so sf_t[c, b] must grow with c; rows b*128.. share a scale per column
    y = np.ones((256, 256), np.float32) * (np.arange(256, dtype=np.float32) + 1)[None, :]
    y[128:] *= 2
    _, st = oracle.cast_cols_f32(y, "e4m3")
    exp0 = (np.arange(256, dtype=np.float32) + 1) / np.float32(448)
    assert np.array_equal(st[:, 0], exp0)
    assert np.array_equal(st[:, 1], ((np.arange(256, dtype=np.float32) + 1) * 2) / np.float32(448))


# ---------------------------------------------------------------------------
# SwiGLU values
# ---------------------------------------------------------------------------

def _swiglu_input(T=64, H=256, seed=17, gate_std=2.0):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((T, H)).astype(np.float32) * np.float32(gate_std)
    u = rng.standard_normal((T, H)).astype(np.float32)
    x = np.concatenate([synth.f32_to_bf16_bits(g), synth.f32_to_bf16_bits(u)], axis=1)
    return x


def test_swiglu_vs_binary64():
    x = _swiglu_input()
    H = x.shape[1] // 2
    w = np.random.default_rng(2).uniform(0.01, 1.0, x.shape[0]).astype(np.float32)
    for ww in (None, w):
        y = oracle.swiglu_values(x, ww).astype(np.float64)
        f = synth.bf16_bits_to_f32(x).astype(np.float64)
        g, u = f[:, :H], f[:, H:]
        ref = g / (1.0 + np.exp(-g)) * u
        if ww is not None:
            ref = ref * ww.astype(np.float64)[:, None]
        tol = 4 * 2.0 ** -24 * np.abs(ref) + 1e-38
        assert np.all(np.abs(y - ref) <= tol)


def test_swiglu_vs_torch_silu():
    x = _swiglu_input(seed=23)
    H = x.shape[1] // 2
    y = oracle.swiglu_values(x)
    f = torch.from_numpy(synth.bf16_bits_to_f32(x))
    ref = (torch.nn.functional.silu(f[:, :H]) * f[:, H:]).numpy().astype(np.float64)
    tol = 8 * 2.0 ** -24 * np.abs(ref) + 1e-38
    assert np.all(np.abs(y.astype(np.float64) - ref) <= tol)


def test_swiglu_orientation_and_special_cases():
    H = 128
    x = np.zeros((3, 2 * H), np.uint16)
    g10 = synth.f32_to_bf16_bits(np.array([10.0], np.float32))[0]
    one = synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    mone = synth.f32_to_bf16_bits(np.array([-1.0], np.float32))[0]
    x[0, 0], x[0, H] = g10, one          # gate 10, up 1 -> silu(10) ~ 9.9995
    x[1, :H], x[1, H:] = 0, mone         # gate 0 -> 0 whatever up is
    x[2, 0], x[2, H] = one, g10          # gate 1, up 10 -> 7.3106
    y = oracle.swiglu_values(x)
    assert abs(y[0, 0] - 10.0 / (1 + math.exp(-10.0))) < 1e-5
    assert abs(y[2, 0] - 10.0 / (1 + math.exp(-1.0))) < 1e-5
    assert np.all(y[1] == 0.0)
    assert np.all(y[0, 1:] == 0.0)


def test_swiglu_weight_one_and_weight_product():
    x = _swiglu_input(seed=31)
    T = x.shape[0]
    y0 = oracle.swiglu_values(x)
    y1 = oracle.swiglu_values(x, np.ones(T, np.float32))
    assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    w = np.random.default_rng(4).uniform(0.01, 1.0, T).astype(np.float32)
    yw = oracle.swiglu_values(x, w)
    assert np.array_equal(yw.view(np.uint32), (y0 * w[:, None]).view(np.uint32))


def test_swiglu_cast_t_consistency():
    x = _swiglu_input(T=256, H=256, seed=41)
    out, sf, out_t, sf_t = oracle.swiglu_cast_t(x)
    o2, s2 = oracle.swiglu_cast(x)
    assert np.array_equal(out, o2) and np.array_equal(sf, s2)
    y = oracle.swiglu_values(x)
    ct, st = oracle.cast_rows_f32(np.ascontiguousarray(y.T))
    assert np.array_equal(out_t, ct) and np.array_equal(sf_t, st)
    # threaded block split gives the same arrays
    t4 = oracle.swiglu_cast_t(x, threads=2)
    for a, b in zip((out, sf, out_t, sf_t), t4):
        assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# SwiGLU clamp ("DeepSeek开源TileKernels..." §3.3: gate clamped from above,
# up clamped on both sides, clamps counted)
# ---------------------------------------------------------------------------

def _bf(v):
    return synth.f32_to_bf16_bits(np.asarray(v, np.float32))


def test_swiglu_clamp_hand_values():
    H, c = 128, 5.0
    x = np.zeros((4, 2 * H), np.uint16)
    x[0, 0], x[0, H] = _bf(10.0), _bf(1.0)      # gate above c -> clamped to c
    x[1, 0], x[1, H] = _bf(-10.0), _bf(1.0)     # gate below -c: gates are not clamped from below
    x[2, 0], x[2, H] = _bf(1.0), _bf(8.0)       # up above c -> c
    x[3, 0], x[3, H] = _bf(1.0), _bf(-8.0)      # up below -c -> -c
    x[3, 1], x[3, H + 1] = _bf(5.0), _bf(-5.0)  # exactly at the bound: unchanged, not counted
    y, n = oracle.swiglu_values(x, clamp=c)
    silu = lambda g: g / (1.0 + math.exp(-g))
    assert abs(y[0, 0] - silu(5.0)) < 1e-5
    assert abs(y[1, 0] - silu(-10.0)) < 1e-9
    assert abs(y[2, 0] - 5.0 * silu(1.0)) < 1e-5
    assert abs(y[3, 0] + 5.0 * silu(1.0)) < 1e-5
    assert abs(y[3, 1] + 5.0 * silu(5.0)) < 1e-4
    assert n == 3


@pytest.mark.parametrize("c", [0.5, 1.5, 3.0])
def test_swiglu_clamp_is_the_swiglu_of_the_clipped_input(c):
    """With a bf16-representable bound, clamping inside the oracle equals the
    unclamped oracle on an input clipped beforehand with numpy, and the count is
    the number of entries np.clip changes."""
    x = _swiglu_input(T=64, H=256, seed=61)
    H = x.shape[1] // 2
    f = synth.bf16_bits_to_f32(x)
    g, u = f[:, :H], f[:, H:]
    clipped = np.concatenate([np.minimum(g, c), np.clip(u, -c, c)], axis=1)
    xc = synth.f32_to_bf16_bits(clipped)
    w = np.random.default_rng(5).uniform(0.01, 1.0, x.shape[0]).astype(np.float32)
    for ww in (None, w):
        y, n = oracle.swiglu_values(x, ww, clamp=c)
        assert np.array_equal(y.view(np.uint32), oracle.swiglu_values(xc, ww).view(np.uint32))
        assert n == int(np.count_nonzero(g > c) + np.count_nonzero(np.abs(u) > c))
    assert n > 0


def test_swiglu_clamp_beyond_the_data_changes_nothing():
    x = _swiglu_input(T=32, H=128, seed=62)
    y0 = oracle.swiglu_values(x)
    y1, n = oracle.swiglu_values(x, clamp=1e30)
    assert n == 0 and np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    with pytest.raises(ValueError):
        oracle.swiglu_values(x, clamp=-1.0)


def test_swiglu_clamp_casts_compose():
    """The clamped casts are the casts of the clamped values; the threaded
    split sums the per-block counts."""
    x = _swiglu_input(T=256, H=256, seed=63)
    y, n = oracle.swiglu_values(x, clamp=1.0)
    out, sf, n1 = oracle.swiglu_cast(x, clamp=1.0)
    o2, s2 = oracle.cast_rows_f32(y)
    assert n1 == n and np.array_equal(out, o2) and np.array_equal(sf, s2)
    res = oracle.swiglu_cast_t(x, clamp=1.0, threads=2)
    ct, st = oracle.cast_rows_f32(np.ascontiguousarray(y.T))
    assert np.array_equal(res[0], o2) and np.array_equal(res[2], ct) and np.array_equal(res[3], st)
    assert res[4] == n


def test_invalid_arguments_raise():
    with pytest.raises(ValueError):
        oracle.per_token_cast(np.zeros((2, 100), np.uint16))
    with pytest.raises(ValueError):
        oracle.swiglu_cast_t(np.zeros((100, 256), np.uint16))


# ---------------------------------------------------------------------------
# SwiGLU backward
# ---------------------------------------------------------------------------

def _bwd_inputs(T=32, H=128, seed=51):
    rng = np.random.default_rng(seed)
    x = _swiglu_input(T, H, seed=seed)
    dy = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    w = rng.uniform(0.01, 1.0, T).astype(np.float32)
    return x, dy, w


def test_swiglu_backward_vs_finite_differences():
    """Central differences of the forward formula g / (1 + exp(-g)) * u * w in
    binary64: independent of the closed-form derivative the oracle uses."""
    x, dy, w = _bwd_inputs()
    H = x.shape[1] // 2
    grad = oracle.swiglu_backward_values(x, dy, w).astype(np.float64)
    f = synth.bf16_bits_to_f32(x).astype(np.float64)
    g, u = f[:, :H], f[:, H:]
    d = synth.bf16_bits_to_f32(dy).astype(np.float64)
    wt = w.astype(np.float64)[:, None]
    y = lambda gg, uu: gg / (1.0 + np.exp(-gg)) * uu * wt
    h = 1e-5
    fd_g = d * (y(g + h, u) - y(g - h, u)) / (2 * h)
    fd_u = d * (y(g, u + h) - y(g, u - h)) / (2 * h)
    scale = np.abs(d * wt) * (np.abs(u) + np.abs(g) + 1.0)
    assert np.all(np.abs(grad[:, :H] - fd_g) <= 1e-6 * scale + 1e-9)
    assert np.all(np.abs(grad[:, H:] - fd_u) <= 1e-6 * scale + 1e-9)


def test_swiglu_backward_vs_torch_autograd():
    x, dy, w = _bwd_inputs(seed=53)
    H = x.shape[1] // 2
    grad = oracle.swiglu_backward_values(x, dy, w).astype(np.float64)
    f = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    g = f[:, :H].clone().requires_grad_(True)
    u = f[:, H:].clone().requires_grad_(True)
    d = torch.from_numpy(synth.bf16_bits_to_f32(dy).astype(np.float64))
    y = torch.nn.functional.silu(g) * u * torch.from_numpy(w.astype(np.float64))[:, None]
    y.backward(d)
    ref = np.concatenate([g.grad.numpy(), u.grad.numpy()], axis=1)
    tol = 2.0 ** -23 * np.abs(ref) + 1e-30
    assert np.all(np.abs(grad - ref) <= tol)


def test_swiglu_backward_special_cases():
    H = 128
    x = np.zeros((3, 2 * H), np.uint16)
    dy = np.zeros((3, H), np.uint16)
    one = synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    three = synth.f32_to_bf16_bits(np.array([3.0], np.float32))[0]
    x[0, H:] = three            # g = 0, u = 3, dy = 1: dg = 0.5 * 3, du = 0
    dy[0] = one
    x[1, :H] = three            # dy = 0 everywhere in row 1: all zero
    x[2, :H] = three            # g = 3, u = 0, dy = 1: dg = 0, du = silu(3)
    dy[2] = one
    grad = oracle.swiglu_backward_values(x, dy)
    assert np.all(grad[0, :H] == 1.5) and np.all(grad[0, H:] == 0)
    assert np.all(grad[1] == 0)
    assert np.all(grad[2, :H] == 0)
    assert np.allclose(grad[2, H:], 3.0 / (1 + math.exp(-3.0)), rtol=1e-7)


def test_swiglu_backward_cast_is_cast_of_values():
    x, dy, w = _bwd_inputs(T=64, H=256, seed=57)
    grad = oracle.swiglu_backward_values(x, dy, w)
    c1, s1 = oracle.cast_rows_f32(grad)
    c2, s2 = oracle.swiglu_backward_cast(x, dy, w)
    assert np.array_equal(c1, c2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


# ---------------------------------------------------------------------------
# scale-factor layout options
# ---------------------------------------------------------------------------

def test_pow2_ceil_against_numpy_and_properties():
    rng = np.random.default_rng(61)
    s = np.concatenate([np.exp2(rng.uniform(-30, 20, 20000)),
                        np.exp2(rng.integers(-30, 20, 200).astype(np.float64))]).astype(np.float32)
    got = np.array([oracle.pow2_ceil(v) for v in s], np.float32)
    ref = np.exp2(np.ceil(np.log2(s.astype(np.float64)))).astype(np.float32)
    assert np.array_equal(got, ref)
    m, _ = np.frexp(got)
    assert np.all(m == 0.5) and np.all(got >= s) and np.all(got < 2 * s)
    exact = np.frexp(s)[0] == 0.5
    assert np.all((got == s) == exact)


def test_round_pow2_codes_are_exact_scaling():
    """With a power-of-two scale 2^k the quotient y / s is exact, so the codes
    are torch's FP8 conversion of y * 2^-k (in range) and the scale is the
    plain scale rounded up."""
    rng = np.random.default_rng(63)
    y = (rng.standard_normal((64, 512)) * np.exp2(rng.integers(-8, 8, (64, 1)))).astype(np.float32)
    for fmt in FMTS:
        c0, s0 = oracle.cast_rows_f32(y, fmt)
        c1, s1 = oracle.cast_rows_f32_ex(y, fmt, 128, oracle.SF_ROUND_POW2)
        assert np.array_equal(s1, np.exp2(np.ceil(np.log2(s0.astype(np.float64)))).astype(np.float32))
        q = y.reshape(64, 4, 128) / s1[:, :, None]
        assert np.all(np.abs(q) <= FMAX[fmt])
        ref = torch.from_numpy(np.ascontiguousarray(q.reshape(64, 512))).to(TORCH_FP8[fmt])
        assert np.array_equal(c1, ref.view(torch.uint8).numpy())


def test_round_pow2_hand_group():
    # amax 3.140625: s0 = fl(3.140625 / 448) ~ 0.00701 -> s = 2^-7; the amax
    # element becomes 402, between 384 and 416 above the midpoint 400 -> 416
    # (0x7d); 1.0 becomes exactly 128 (0x70).
    y = np.zeros((1, 128), np.float32)
    y[0, 3], y[0, 9] = 3.140625, 1.0
    c, s = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.SF_ROUND_POW2)
    assert s[0, 0] == np.float32(2.0 ** -7)
    assert c[0, 3] == 0x7D and c[0, 9] == 0x70 and np.count_nonzero(c) == 2
    c, s = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.SF_UE8M0_PACKED)
    assert s.dtype == np.uint32 and s[0, 0] == 127 - 7   # one group: byte 0 only


def test_reciprocal_reading_hand_groups():
    """The reciprocal-multiply reading (codes of fl32(v * fl32(1 / s))): the two
    quotient-tie groups give their hand-worked codes_reciprocal (one step away
    from the quotient's codes); every group whose scale is a power of two,
    where the product by the reciprocal is the exact quotient, keeps the
    quotient's codes; the scales never change."""
    spec = json.load(open(os.path.join(GOLDEN, "hand_groups.json")))
    G = spec["group"]
    seen = 0
    for case in spec["cases"]:
        vals = np.full(G, case["fill"], np.float32)
        for k, v in case["set"].items():
            vals[int(k)] = np.float32(v)
        y = vals.reshape(1, G)
        codes, sf = oracle.cast_rows_f32_ex(y, case["fmt"], G, oracle.Q_RECIPROCAL)
        assert hex(int(sf.view(np.uint32)[0, 0])) == case["scale_hex"], case["name"]
        scale_bits = int(case["scale_hex"], 16)
        if "codes_reciprocal" in case:
            want = case["codes_reciprocal"]
            seen += 1
        elif scale_bits & 0x007FFFFF == 0:
            want = case["codes"]
        else:
            continue
        exp = np.full(G, int(case["code_fill"], 16), np.uint8)
        for k, c in want.items():
            exp[int(k)] = int(c, 16)
        bad = np.nonzero(codes[0] != exp)[0]
        assert bad.size == 0, (case["name"], [(int(i), hex(codes[0, i]), hex(exp[i])) for i in bad])
    assert seen == 2


@pytest.mark.parametrize("fmt", FMTS)
def test_reciprocal_reading_properties(fmt):
    """On seeded data: with power-of-two scales both readings give the same
    codes; otherwise a code differs from the quotient's by at most one FP8 step
    (the product is within about one binary32 ulp of the quotient), and the
    scales are those of the quotient reading."""
    y = _layout_inputs(T=64, G=8, seed=71)
    c_q, s_q = oracle.cast_rows_f32_ex(y, fmt, 128, 0)
    c_r, s_r = oracle.cast_rows_f32_ex(y, fmt, 128, oracle.Q_RECIPROCAL)
    assert np.array_equal(s_q, s_r)
    # one step: adjacent codes of the same sign (the byte order of FP8 codes
    # follows the magnitude within a sign)
    same_sign = (c_q & 0x80) == (c_r & 0x80)
    step = np.abs((c_q & 0x7F).astype(int) - (c_r & 0x7F).astype(int))
    assert np.all(same_sign | ((c_q & 0x7F) == 0) & ((c_r & 0x7F) == 0))
    assert step.max() <= 1
    for flags in (oracle.SF_ROUND_POW2, oracle.SF_UE8M0_PACKED | oracle.SF_COL_MAJOR):
        c1, s1 = oracle.cast_rows_f32_ex(y, fmt, 128, flags)
        c2, s2 = oracle.cast_rows_f32_ex(y, fmt, 128, flags | oracle.Q_RECIPROCAL)
        assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_unknown_flag_is_rejected():
    with pytest.raises(Exception):
        oracle.cast_rows_f32_ex(np.zeros((1, 128), np.float32), "e4m3", 128, 16)


def _layout_inputs(T=13, G=7, seed=67):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, G * 128)) * np.exp2(rng.integers(-6, 6, (T, G * 128))
                                                         )).astype(np.float32)


@pytest.mark.parametrize("flags", [oracle.SF_COL_MAJOR, oracle.SF_UE8M0_PACKED,
                                   oracle.SF_UE8M0_PACKED | oracle.SF_COL_MAJOR,
                                   oracle.SF_ROUND_POW2 | oracle.SF_COL_MAJOR])
def test_sf_layouts_rearrange_the_row_major_scales(flags):
    y = _layout_inputs()
    T, C = y.shape
    G = C // 128
    pow2 = flags & (oracle.SF_ROUND_POW2 | oracle.SF_UE8M0_PACKED)
    c_ref, s_ref = oracle.cast_rows_f32_ex(y, "e4m3", 128, oracle.SF_ROUND_POW2 if pow2 else 0)
    c, s = oracle.cast_rows_f32_ex(y, "e4m3", 128, flags)
    assert np.array_equal(c, c_ref)
    T4 = (T + 3) // 4 * 4
    if flags & oracle.SF_UE8M0_PACKED:
        e = ((s_ref.view(np.uint32) >> 23) & 0xFF).astype(np.uint32)
        assert np.array_equal(np.exp2(e.astype(np.float64) - 127).astype(np.float32), s_ref)
        W = (G + 3) // 4
        ep = np.zeros((T, W * 4), np.uint32)
        ep[:, :G] = e
        words = ep[:, 0::4] | (ep[:, 1::4] << 8) | (ep[:, 2::4] << 16) | (ep[:, 3::4] << 24)
        if flags & oracle.SF_COL_MAJOR:
            assert s.shape == (W, T4)
            assert np.array_equal(s[:, :T], words.T) and np.all(s[:, T:] == 0)
        else:
            assert np.array_equal(s, words)
    else:
        assert s.shape == (G, T4)
        assert np.array_equal(s[:, :T], s_ref.T) and np.all(s[:, T:] == 0)


# ---------------------------------------------------------------------------
# per-channel / per-block casts, cast back
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FMTS)
def test_per_channel_is_per_token_of_transpose(fmt):
    x = _random_bits(T=256, C=384, seed=71)
    xt = np.ascontiguousarray(x.T)
    ct, st = oracle.per_token_cast(xt, fmt)            # [C, T], [C, T/128]
    c1, s1 = oracle.per_channel_cast(x, fmt, 128, transpose=True)
    assert np.array_equal(c1, ct) and np.array_equal(s1.view(np.uint32), st.view(np.uint32))
    c0, s0 = oracle.per_channel_cast(x, fmt, 128, transpose=False)
    assert np.array_equal(c0, ct.T) and np.array_equal(s0.view(np.uint32), st.T.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("T", [256, 300])
def test_per_block_is_per_token_of_flattened_blocks(fmt, T):
    """Each 128 x 128 block flattened into one row of 16384 values is one group
    of the per-token cast (group = 16384; the short last block: rows * 128)."""
    x = _random_bits(T=T, C=384, seed=73)
    codes, sf = oracle.per_block_cast(x, fmt, 128)
    for rb in range(-(-T // 128)):
        r0, r1 = rb * 128, min(T, rb * 128 + 128)
        for cb in range(3):
            blk = np.ascontiguousarray(x[r0:r1, cb * 128:(cb + 1) * 128]).reshape(1, -1)
            c, s = oracle.per_token_cast(blk, fmt, group=blk.shape[1])
            assert s[0, 0] == sf[rb, cb]
            assert np.array_equal(c.reshape(r1 - r0, 128), codes[r0:r1, cb * 128:(cb + 1) * 128])


@pytest.mark.parametrize("fmt", FMTS)
def test_cast_back_matches_torch_decode(fmt):
    x = _random_bits(T=64, C=512, seed=79)
    codes, sf = oracle.per_token_cast(x, fmt)
    y = oracle.cast_back(codes, sf, 1, 128, fmt)
    dec = torch.from_numpy(codes).view(TORCH_FP8[fmt]).to(torch.float32).numpy()
    ref = dec * np.repeat(sf, 128, axis=1)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))
    # round trip within half an FP8 step of each value, plus the binary32
    # rounding of the quotient (it may land exactly on an FP8 tie and then go
    # the even way) and of the product decode * s
    v = synth.bf16_bits_to_f32(x).astype(np.float64)
    s = np.repeat(sf.astype(np.float64), 128, axis=1)
    q = np.abs(v / s)
    e = np.maximum(np.floor(np.log2(np.maximum(q, 1e-300))), EMIN[fmt])
    bound = 0.5 * np.exp2(e - MBITS[fmt]) * s + q * s * 2.0 ** -23 + np.abs(v) * 2.0 ** -23
    assert np.all(np.abs(y - v) <= bound + 1e-30)


def test_cast_back_hand_values_and_granularities():
    codes = np.zeros((256, 256), np.uint8)
    codes[0, 0], codes[200, 130] = 0x7E, 0x01          # 448, 2^-9 (E4M3)
    sf_tok = np.ones((256, 2), np.float32)
    sf_tok[200, 1] = 2.0
    y = oracle.cast_back(codes, sf_tok, 1, 128, "e4m3")
    assert y[0, 0] == 448.0 and y[200, 130] == 2.0 ** -8 and np.count_nonzero(y) == 2
    sf_blk = np.array([[0.5, 1.0], [1.0, 4.0]], np.float32)    # 128 x 128 blocks
    y = oracle.cast_back(codes, sf_blk, 128, 128, "e4m3")
    assert y[0, 0] == 224.0 and y[200, 130] == 2.0 ** -7
    sf_ch = np.ones((2, 256), np.float32)
    sf_ch[1, 130] = 8.0                                        # 128 x 1 groups
    y = oracle.cast_back(codes, sf_ch, 128, 1, "e4m3")
    assert y[200, 130] == 2.0 ** -6
