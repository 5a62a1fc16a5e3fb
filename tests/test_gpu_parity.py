"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

* plain cast: codes and scales bit-exact, at the workloads' full sizes, ragged
  shapes, tie-heavy inputs, every bf16 value, hand-worked groups, and an input
  of more than 2^31 elements (sampled rows);
* SwiGLU cast (+ routing weight): scales within 1e-6 relative, codes within one
  FP8 step with at most 1e-4 differing, at full sizes and ragged shapes;
* SwiGLU + transposed cast: the same tolerance for both outputs, row outputs
  bit-identical to the SwiGLU cast; at full size on sampled token blocks.
Every output buffer is surrounded by guard bytes that must stay untouched.
"""
from __future__ import annotations

import ctypes
import json
import os

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))
GUARD = 256
GUARD_BYTE = 0xA5
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


class Guarded:
    """A device byte buffer with GUARD bytes of a known pattern on both sides."""

    def __init__(self, nbytes: int, dev):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), GUARD_BYTE, dtype=torch.uint8, device=dev)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + GUARD)

    def data(self) -> np.ndarray:
        return self.buf[GUARD:GUARD + self.n].cpu().numpy()

    def check_guards(self, name):
        h = self.buf.cpu().numpy()
        assert np.all(h[:GUARD] == GUARD_BYTE) and np.all(h[GUARD + self.n:] == GUARD_BYTE), \
            f"{name}: write outside the output buffer"


def to_dev_bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def stream_of(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def run_plain(x_bits, fmt, dev):
    T, C = x_bits.shape
    xd = to_dev_bf16(x_bits, dev)
    out = Guarded(T * C, dev)
    sf = Guarded(T * (C // 128) * 4, dev)
    st = tkq.tkq_per_token_cast(ctypes.c_void_p(xd.data_ptr()), out.ptr, sf.ptr, T, C, 128,
                                oracle.FMT[fmt], stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    return out.data().reshape(T, C), sf.data().view(np.float32).reshape(T, C // 128)


def run_swiglu(x_bits, w, fmt, dev, transposed=False):
    T, H2 = x_bits.shape
    H = H2 // 2
    xd = to_dev_bf16(x_bits, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    wp = None if wd is None else ctypes.c_void_p(wd.data_ptr())
    out = Guarded(T * H, dev)
    sf = Guarded(T * (H // 128) * 4, dev)
    if not transposed:
        st = tkq.tkq_swiglu_cast(ctypes.c_void_p(xd.data_ptr()), wp, out.ptr, sf.ptr, T, H, 128,
                                 oracle.FMT[fmt], stream_of(dev))
        assert st == 0, tkq.tkq_status_string(st)
        torch.cuda.synchronize()
        out.check_guards("out")
        sf.check_guards("sf")
        return out.data().reshape(T, H), sf.data().view(np.float32).reshape(T, H // 128)
    out_t = Guarded(T * H, dev)
    sf_t = Guarded(H * (T // 128) * 4, dev)
    st = tkq.tkq_swiglu_cast_t(ctypes.c_void_p(xd.data_ptr()), wp, out.ptr, sf.ptr, out_t.ptr,
                               sf_t.ptr, T, H, 128, oracle.FMT[fmt], stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    for g, n in ((out, "out"), (sf, "sf"), (out_t, "out_t"), (sf_t, "sf_t")):
        g.check_guards(n)
    return (out.data().reshape(T, H), sf.data().view(np.float32).reshape(T, H // 128),
            out_t.data().reshape(H, T), sf_t.data().view(np.float32).reshape(H, T // 128))


# ---------------------------------------------------------------------------
# plain cast: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,fmt", [("plain_small", "e4m3"), ("plain_outlier", "e4m3"),
                                      ("plain_outlier", "e5m2")])
def test_plain_cast_full_workload(cuda_device, name, fmt):
    x = synth.workload(name)["x"]
    out, sf = run_plain(x, fmt, cuda_device)
    ro, rs = oracle.per_token_cast(x, fmt, threads=THREADS)
    parity.assert_bit_exact(f"{name} {fmt} scales", sf, rs)
    parity.assert_bit_exact(f"{name} {fmt} codes", out, ro)


@pytest.mark.parametrize("T", [1, 7, 129, 8191])
@pytest.mark.parametrize("C", [128, 256, 384, 7168])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_plain_cast_ragged(cuda_device, T, C, fmt):
    x =synth.workload("plain_outlier", rows=T)["x"][:, :C].copy()
    out, sf = run_plain(x, fmt, cuda_device)
    ro, rs = oracle.per_token_cast(x, fmt, threads=THREADS)
    parity.assert_bit_exact("scales", sf, rs)
    parity.assert_bit_exact("codes", out, ro)


def _tie_heavy_bits(T, C, seed):
    """bf16 values with 1-4 significant bits: their quotients by the group scale
    often land exactly on FP8 rounding ties (e.g. 0.97265625 / 2.59375 = 0.375)."""
    rng = np.random.default_rng(seed)
    mant = rng.integers(1, 16, size=(T, C)).astype(np.float32)
    exp = rng.integers(-12, 4, size=(T, C)).astype(np.float32)
    sign = np.where(rng.random((T, C)) < 0.5, -1.0, 1.0).astype(np.float32)
    v = sign * mant * np.exp2(exp).astype(np.float32)
    return synth.f32_to_bf16_bits(v)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_plain_cast_tie_heavy(cuda_device, fmt):
    x = _tie_heavy_bits(2048, 2048, seed=5)
    out, sf = run_plain(x, fmt, cuda_device)
    ro, rs = oracle.per_token_cast(x, fmt, threads=THREADS)
    parity.assert_bit_exact("scales", sf, rs)
    parity.assert_bit_exact("codes", out, ro)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_plain_cast_every_bf16_value(cuda_device, fmt):
    """Groups [fmt_max, v1 .. v127] have scale exactly 1, so the codes are the
    FP8 conversions of every finite bf16 value of magnitude <= fmt_max."""
    fmax = 448.0 if fmt == "e4m3" else 57344.0
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(allb)
    vals = allb[np.isfinite(f) & (np.abs(f) <= fmax)]
    n = -(-vals.size // 127)
    body = np.zeros(n * 127, np.uint16)
    body[:vals.size] = vals
    head = synth.f32_to_bf16_bits(np.full((n, 1), fmax, np.float32))
    x = np.concatenate([head, body.reshape(n, 127)], axis=1)
    out, sf = run_plain(x, fmt, cuda_device)
    assert np.all(sf == 1.0)
    ro, rs = oracle.per_token_cast(x, fmt, threads=THREADS)
    parity.assert_bit_exact("codes", out, ro)


def test_plain_cast_hand_groups(cuda_device):
    spec = json.load(open(os.path.join(GOLDEN, "hand_groups.json")))
    for case in spec["cases"]:
        vals = np.full(128, case["fill"], np.float32)
        for k, v in case["set"].items():
            vals[int(k)] = np.float32(v)
        x = synth.f32_to_bf16_bits(vals).reshape(1, 128)
        out, sf = run_plain(x, case["fmt"], cuda_device)
        assert hex(int(sf.view(np.uint32)[0, 0])) == case["scale_hex"], case["name"]
        exp = np.full(128, int(case["code_fill"], 16), np.uint8)
        for k, c in case["codes"].items():
            exp[int(k)] = int(c, 16)
        parity.assert_bit_exact(case["name"], out[0], exp)


@pytest.mark.slow
def test_plain_cast_beyond_2_31_elements(cuda_device):
    """x of 524,293 x 4096 bf16 (2.15e9 elements, 4.3 GB): byte offsets beyond
    2^32; rows sampled at both ends and the middle are checked bit-exact."""
    T, C = 524_293, 4096
    dev = cuda_device
    rng = np.random.default_rng(77)
    xd = torch.empty((T, C), dtype=torch.int16, device=dev)
    chunk = 65536
    keep = {}
    sample_rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(T - 300, T),
                                            rng.integers(0, T, 64)]))
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        bits = rng.integers(0, 1 << 16, size=(b - a, C), dtype=np.uint16)
        # keep sign and mantissa, put the exponent in a finite, moderate range
        e = rng.integers(127 - 20, 127 + 12, size=(b - a, C), dtype=np.uint16)
        bits = (bits & np.uint16(0x807F)) | (e << np.uint16(7)).astype(np.uint16)
        xd[a:b] = torch.from_numpy(bits.view(np.int16)).to(dev)
        sel = sample_rows[(sample_rows >= a) & (sample_rows < b)]
        for r in sel:
            keep[int(r)] = bits[r - a].copy()
    out = torch.empty((T, C), dtype=torch.uint8, device=dev)
    sf = torch.empty((T, C // 128), dtype=torch.float32, device=dev)
    st = tkq.tkq_per_token_cast(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(sf.data_ptr()), T, C, 128, 0, stream_of(dev))
    assert st == 0
    torch.cuda.synchronize()
    rows = np.array(sorted(keep))
    xs = np.stack([keep[r] for r in rows])
    ro, rs = oracle.per_token_cast(xs, "e4m3", threads=THREADS)
    idx = torch.from_numpy(rows).to(dev)
    parity.assert_bit_exact("codes", out.index_select(0, idx).cpu().numpy(), ro)
    parity.assert_bit_exact("scales", sf.index_select(0, idx).cpu().numpy(), rs)


# ---------------------------------------------------------------------------
# SwiGLU cast: tolerance
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["swiglu", "swiglu_moe"])
def test_swiglu_full_workload(cuda_device, name):
    d = synth.workload(name)
    w = d.get("w")
    out, sf = run_swiglu(d["x"], w, "e4m3", cuda_device)
    ro, rs = oracle.swiglu_cast(d["x"], w, "e4m3", threads=THREADS)
    parity.assert_scales_close("scales", sf, rs)
    parity.assert_codes_close("codes", out, ro)


@pytest.mark.parametrize("T", [1, 7, 129, 1031])
@pytest.mark.parametrize("H", [128, 384, 2048])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_swiglu_ragged(cuda_device, swiglu_kernel, T, H, weighted, fmt):
    d = synth.workload("swiglu_moe", rows=T)
    x = np.ascontiguousarray(d["x"][:, np.r_[0:H, 2048:2048 + H]])
    w = d["w"] if weighted else None
    out, sf = run_swiglu(x, w, fmt, cuda_device)
    ro, rs = oracle.swiglu_cast(x, w, fmt, threads=THREADS)
    parity.assert_scales_close("scales", sf, rs)
    # small cases: allow a single differing code below the 1e-4 fraction
    parity.assert_codes_close("codes", out, ro, max_frac=max(1e-4, 1.0 / out.size))


def test_swiglu_gate_orientation_and_zero_gate(cuda_device, swiglu_kernel):
    H = 128
    x = np.zeros((2, 2 * H), np.uint16)
    x[0, :H] = synth.f32_to_bf16_bits(np.full(H, 10.0, np.float32))
    x[0, H:] = synth.f32_to_bf16_bits(np.linspace(-2, 2, H).astype(np.float32))
    x[1, H:] = synth.f32_to_bf16_bits(np.full(H, -3.0, np.float32))  # gate 0 -> y = -0
    out, sf = run_swiglu(x, None, "e4m3", cuda_device)
    ro, rs = oracle.swiglu_cast(x, None, "e4m3")
    parity.assert_scales_close("scales", sf, rs)
    parity.assert_codes_close("codes", out, ro, max_frac=1.0 / out.size)
    assert np.all(out[1] == 0x80)  # -0 keeps its sign


@pytest.mark.parametrize("flags", [0, 1, 4, 6])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("clamp", [None, 2.0, 2.9])
@pytest.mark.parametrize("T,H", [(1031, 384), (4099, 2048)])
def test_swiglu_kernels_agree_bytewise(cuda_device, monkeypatch, flags, weighted, clamp, T, H):
    """The flat and the TMA-ring SwiGLU kernels give the same bytes (codes,
    scales in every layout, clamp count) on the same input: the library may
    pick either for a call."""
    d = synth.workload("swiglu_moe", rows=T)
    x = np.ascontiguousarray(d["x"][:, np.r_[0:H, 2048:2048 + H]])
    xd = to_dev_bf16(x, cuda_device)
    w = torch.from_numpy(d["w"]).to(cuda_device) if weighted else None
    opts = dict(round_sf=bool(flags & 1), use_packed_ue8m0=bool(flags & 2),
                use_tma_aligned_col_major_sf=bool(flags & 4))
    got = {}
    for kernel in ("flat", "ring"):
        monkeypatch.setenv("TKQ_SWIGLU_KERNEL", kernel)
        cnt = torch.zeros(1, dtype=torch.int64, device=cuda_device)
        kw = dict(use_clamp=True, swiglu_clamp_value=clamp, clamp_count=cnt) if clamp else {}
        q, s = tkq.swiglu_forward_and_per_token_cast(xd, topk_weights=w, **opts, **kw)
        got[kernel] = [q.view(torch.uint8).cpu().numpy(), s.contiguous().view(torch.uint8).cpu().numpy(),
                       cnt.cpu().numpy()]
    for a, b, what in zip(got["flat"], got["ring"], ("codes", "scales", "clamp count")):
        parity.assert_bit_exact(what, a, b)
    assert tkq.tkq_read_device_status() == 0


def test_swiglu_beyond_2_31_input_elements(cuda_device, monkeypatch):
    """x of 262,147 x 8192 bf16 (2.15e9 elements, 4.3 GB) with a routing
    weight, through both SwiGLU kernels: input offsets beyond 2^32 bytes.  The
    two outputs are compared byte for byte in full, and rows sampled at both
    ends and the middle against the oracle."""
    T, H = 262_147, 4096
    dev = cuda_device
    rng = np.random.default_rng(78)
    xd = torch.empty((T, 2 * H), dtype=torch.int16, device=dev)
    w = rng.uniform(0.0, 1.0, T).astype(np.float32)
    wd = torch.from_numpy(w).to(dev)
    chunk = 32768
    keep = {}
    sample_rows = np.unique(np.concatenate([np.arange(0, 32), np.arange(T - 200, T),
                                            rng.integers(0, T, 48)]))
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        bits = rng.integers(0, 1 << 16, size=(b - a, 2 * H), dtype=np.uint16)
        e = rng.integers(127 - 8, 127 + 3, size=(b - a, 2 * H), dtype=np.uint16)
        bits = (bits & np.uint16(0x807F)) | (e << np.uint16(7)).astype(np.uint16)
        xd[a:b] = torch.from_numpy(bits.view(np.int16)).to(dev)
        sel = sample_rows[(sample_rows >= a) & (sample_rows < b)]
        for r in sel:
            keep[int(r)] = bits[r - a].copy()
    got = {}
    for kernel in ("flat", "ring"):
        monkeypatch.setenv("TKQ_SWIGLU_KERNEL", kernel)
        out = torch.empty((T, H), dtype=torch.uint8, device=dev)
        sf = torch.empty((T, H // 128), dtype=torch.float32, device=dev)
        st = tkq.tkq_swiglu_cast(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(wd.data_ptr()),
                                 ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
                                 T, H, 128, 0, stream_of(dev))
        assert st == 0
        torch.cuda.synchronize()
        got[kernel] = (out, sf)
    assert torch.equal(got["flat"][0], got["ring"][0]), "codes of the two kernels differ"
    assert torch.equal(got["flat"][1].view(torch.int32), got["ring"][1].view(torch.int32))
    rows = np.array(sorted(keep))
    xs = np.stack([keep[r] for r in rows])
    ro, rs = oracle.swiglu_cast(xs, w[rows], "e4m3", threads=THREADS)
    idx = torch.from_numpy(rows).to(dev)
    out, sf = got["flat"]
    parity.assert_scales_close("scales", sf.index_select(0, idx).cpu().numpy(), rs)
    codes = out.index_select(0, idx).cpu().numpy()
    parity.assert_codes_close("codes", codes, ro, max_frac=max(1e-4, 1.0 / codes.size))
    assert tkq.tkq_read_device_status() == 0


# ---------------------------------------------------------------------------
# SwiGLU + transposed cast
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,H", [(128, 128), (256, 384), (1024, 2048), (3072, 256)])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_swiglu_t_shapes(cuda_device, swiglu_kernel, T, H, weighted, fmt):
    d = synth.workload("swiglu_moe", rows=T)
    x = np.ascontiguousarray(d["x"][:, np.r_[0:H, 2048:2048 + H]])
    w = d["w"] if weighted else None
    out, sf, out_t, sf_t = run_swiglu(x, w, fmt, cuda_device, transposed=True)
    ro, rs, rot, rst = oracle.swiglu_cast_t(x, w, fmt, threads=THREADS)
    lim = max(1e-4, 1.0 / out.size)
    parity.assert_scales_close("row scales", sf, rs)
    parity.assert_codes_close("row codes", out, ro, max_frac=lim)
    parity.assert_scales_close("column scales", sf_t, rst)
    parity.assert_codes_close("column codes", out_t, rot, max_frac=lim)
    o2, s2 = run_swiglu(x, w, fmt, cuda_device)
    parity.assert_bit_exact("rows of _t == swiglu_cast rows", out, o2)
    parity.assert_bit_exact("row scales of _t == swiglu_cast", sf, s2)


@pytest.mark.slow
def test_swiglu_t_full_workload(cuda_device):
    """The full [131072, 4096] workload in the launch the benchmark times:
    every row and column output against the oracle (all 2 x 268 M codes and
    their scales), and every row output against the SwiGLU cast kernel bit
    for bit."""
    dev = cuda_device
    x = synth.workload("swiglu_t")["x"]
    T, H2 = x.shape
    H = H2 // 2
    xd = to_dev_bf16(x, dev)
    out = torch.empty((T, H), dtype=torch.uint8, device=dev)
    sf = torch.empty((T, H // 128), dtype=torch.float32, device=dev)
    out_t = torch.empty((H, T), dtype=torch.uint8, device=dev)
    sf_t = torch.empty((H, T // 128), dtype=torch.float32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = tkq.tkq_swiglu_cast_t(p(xd), None, p(out), p(sf), p(out_t), p(sf_t), T, H, 128, 0,
                               stream_of(dev))
    assert st == 0
    out2 = torch.empty_like(out)
    sf2 = torch.empty_like(sf)
    st = tkq.tkq_swiglu_cast(p(xd), None, p(out2), p(sf2), T, H, 128, 0, stream_of(dev))
    assert st == 0
    torch.cuda.synchronize()
    assert tkq.tkq_read_device_status() == 0, "a bounded wait gave up"
    assert torch.equal(out, out2) and torch.equal(sf.view(torch.int32), sf2.view(torch.int32))
    del out2, sf2, xd
    ro, rs, rot, rst = oracle.swiglu_cast_t(x, None, "e4m3", threads=THREADS)
    parity.assert_scales_close("row scales", sf.cpu().numpy(), rs)
    parity.assert_codes_close("row codes", out.cpu().numpy(), ro)
    del ro, rs
    parity.assert_scales_close("column scales", sf_t.cpu().numpy(), rst)
    parity.assert_codes_close("column codes", out_t.cpu().numpy(), rot)


# ---------------------------------------------------------------------------
# SwiGLU backward + cast: tolerance
# ---------------------------------------------------------------------------

def run_swiglu_bwd(x_bits, dy_bits, w, fmt, dev):
    T, H2 = x_bits.shape
    H = H2 // 2
    xd = to_dev_bf16(x_bits, dev)
    dyd = to_dev_bf16(dy_bits, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    wp = None if wd is None else ctypes.c_void_p(wd.data_ptr())
    out = Guarded(T * 2 * H, dev)
    sf = Guarded(T * (2 * H // 128) * 4, dev)
    st = tkq.tkq_swiglu_backward_cast(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(dyd.data_ptr()),
                                      wp, out.ptr, sf.ptr, T, H, 128, oracle.FMT[fmt],
                                      stream_of(dev))
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    return out.data().reshape(T, 2 * H), sf.data().view(np.float32).reshape(T, 2 * H // 128)


def test_swiglu_backward_full_workload(cuda_device):
    d = synth.workload("swiglu_bwd")
    out, sf = run_swiglu_bwd(d["x"], d["dy"], d["w"], "e4m3", cuda_device)
    ro, rs = oracle.swiglu_backward_cast(d["x"], d["dy"], d["w"], "e4m3", threads=THREADS)
    parity.assert_scales_close("scales", sf, rs)
    parity.assert_codes_close("codes", out, ro)
    assert tkq.tkq_read_device_status() == 0


@pytest.mark.parametrize("T", [1, 7, 129, 1031])
@pytest.mark.parametrize("H", [128, 384])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_swiglu_backward_ragged(cuda_device, T, H, weighted, fmt):
    d = synth.workload("swiglu_bwd", rows=T)
    x = np.ascontiguousarray(d["x"][:, np.r_[0:H, 2048:2048 + H]])
    dy = np.ascontiguousarray(d["dy"][:, :H])
    w = d["w"] if weighted else None
    out, sf = run_swiglu_bwd(x, dy, w, fmt, cuda_device)
    ro, rs = oracle.swiglu_backward_cast(x, dy, w, fmt, threads=THREADS)
    parity.assert_scales_close("scales", sf, rs)
    parity.assert_codes_close("codes", out, ro, max_frac=max(1e-4, 1.0 / out.size))


def test_swiglu_backward_extreme_gates(cuda_device):
    """Gates from -120 to 120 (exp(-g) overflows binary32 below -88) and of
    magnitude up to 1e38: the gradients must stay finite and match the oracle
    (sigma -> 0 makes both exactly 0 for very negative gates; an exponent
    clamped at 126 would leave dg = d u 2^-126 (1 + g) there, which the codes
    of rows holding gates near -1e38 show)."""
    T, H = 256, 256
    rng = np.random.default_rng(8)
    n = T * H // 2
    big = np.logspace(2.0, 38.0, n // 2) * np.where(np.arange(n // 2) % 2, 1.0, -1.0)
    g = np.concatenate([np.linspace(-120, 120, n), big, -big]).astype(np.float32).reshape(T, H)
    u = rng.standard_normal((T, H)).astype(np.float32)
    x = np.concatenate([synth.f32_to_bf16_bits(g), synth.f32_to_bf16_bits(u)], axis=1)
    dy = synth.f32_to_bf16_bits(rng.uniform(-1.0, 1.0, (T, H)).astype(np.float32))
    out, sf = run_swiglu_bwd(x, dy, None, "e4m3", cuda_device)
    ro, rs = oracle.swiglu_backward_cast(x, dy, None, "e4m3")
    assert np.all(np.isfinite(sf))
    parity.assert_scales_close("scales", sf, rs)
    parity.assert_codes_close("codes", out, ro, max_frac=max(1e-4, 2.0 / out.size))


def test_swiglu_backward_tensor_api(cuda_device):
    d = synth.workload("swiglu_bwd", rows=256)
    x = to_dev_bf16(d["x"], cuda_device)
    dy = to_dev_bf16(d["dy"], cuda_device)
    out, sf = tkq.swiglu_backward_and_per_token_cast(x, dy, "e4m3")
    assert out.dtype == torch.float8_e4m3fn and out.shape == (256, 4096) and sf.shape == (256, 32)
    with pytest.raises(ValueError):
        tkq.swiglu_backward_and_per_token_cast(x, dy[:, :1024].contiguous())


# ---------------------------------------------------------------------------
# scale-factor layouts
# ---------------------------------------------------------------------------

# 8 = TKQ_Q_RECIPROCAL: codes of the product by fl32(1/s) (scales unchanged)
SF_FLAG_SETS = [0, 1, 2, 4, 5, 6, 8, 12, 14]


def sf_rowmajor(raw: np.ndarray, T: int, G: int, flags: int) -> np.ndarray:
    """Any scale layout (raw bytes) -> fp32 [T, G] (test-side decoding)."""
    T4 = (T + 3) // 4 * 4
    W = (G + 3) // 4
    if flags & 2:
        words = raw.view(np.uint32).reshape((W, T4) if flags & 4 else (T, W))
        if flags & 4:
            words = np.ascontiguousarray(words.T[:T])
        b = words.view(np.uint8).reshape(T, W * 4)[:, :G].astype(np.float64)
        return np.exp2(b - 127).astype(np.float32)
    s = raw.view(np.float32).reshape((G, T4) if flags & 4 else (T, G))
    return np.ascontiguousarray(s.T[:T] if flags & 4 else s)


def run_ex(kind, x_bits, flags, fmt, dev, w=None, dy_bits=None):
    T = x_bits.shape[0]
    if kind == "plain":
        C_out, G = x_bits.shape[1], x_bits.shape[1] // 128
    elif kind == "swiglu":
        C_out, G = x_bits.shape[1] // 2, x_bits.shape[1] // 256
    else:
        C_out, G = x_bits.shape[1], x_bits.shape[1] // 128
    xd = to_dev_bf16(x_bits, dev)
    out = Guarded(T * C_out, dev)
    nbytes = tkq.tkq_sf_bytes(T, G, flags)
    sf = Guarded(nbytes, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    wp = None if wd is None else ctypes.c_void_p(wd.data_ptr())
    s = stream_of(dev)
    fc = oracle.FMT[fmt]
    if kind == "plain":
        st = tkq.tkq_per_token_cast_ex(ctypes.c_void_p(xd.data_ptr()), out.ptr, sf.ptr, T, C_out,
                                       128, fc, flags, s)
    elif kind == "swiglu":
        st = tkq.tkq_swiglu_cast_ex(ctypes.c_void_p(xd.data_ptr()), wp, out.ptr, sf.ptr, T, C_out,
                                    128, fc, flags, s)
    else:
        dyd = to_dev_bf16(dy_bits, dev)
        st = tkq.tkq_swiglu_backward_cast_ex(ctypes.c_void_p(xd.data_ptr()),
                                             ctypes.c_void_p(dyd.data_ptr()), wp, out.ptr, sf.ptr,
                                             T, C_out // 2, 128, fc, flags, s)
    assert st == 0, tkq.tkq_status_string(st)
    torch.cuda.synchronize()
    out.check_guards("out")
    sf.check_guards("sf")
    return out.data().reshape(T, C_out), sf.data(), G


@pytest.mark.parametrize("flags", SF_FLAG_SETS)
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_plain_cast_sf_layouts_bit_exact(cuda_device, flags, fmt):
    # G = 7 groups (a partly used last packed word), T = 1031 (padding rows)
    x = synth.workload("plain_outlier", rows=1031)["x"][:, :896].copy()
    out, raw, G = run_ex("plain", x, flags, fmt, cuda_device)
    ro, rs = oracle.per_token_cast_ex(x, fmt, 128, flags, threads=THREADS)
    parity.assert_bit_exact("codes", out, ro)
    parity.assert_bit_exact("scales (raw layout bytes)", raw, rs.view(np.uint8).ravel())


def test_plain_cast_hand_groups_reciprocal(cuda_device):
    """TKQ_Q_RECIPROCAL on the hand-worked groups: the two quotient-tie groups
    give their hand-worked reciprocal codes (0xf3, 0xfb instead of 0xf2, 0xfa);
    groups with a power-of-two scale keep the quotient's codes."""
    spec = json.load(open(os.path.join(GOLDEN, "hand_groups.json")))
    seen = 0
    for case in spec["cases"]:
        vals = np.full(128, case["fill"], np.float32)
        for k, v in case["set"].items():
            vals[int(k)] = np.float32(v)
        x = synth.f32_to_bf16_bits(vals).reshape(1, 128)
        out, raw, _ = run_ex("plain", x, 8, case["fmt"], cuda_device)
        assert hex(int(raw.view(np.uint32)[0])) == case["scale_hex"], case["name"]
        if "codes_reciprocal" in case:
            want = case["codes_reciprocal"]
            seen += 1
        elif int(case["scale_hex"], 16) & 0x007FFFFF == 0:
            want = case["codes"]
        else:
            continue
        exp = np.full(128, int(case["code_fill"], 16), np.uint8)
        for k, c in want.items():
            exp[int(k)] = int(c, 16)
        parity.assert_bit_exact(case["name"], out[0], exp)
    assert seen == 2


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_plain_cast_reciprocal_full_workload(cuda_device, fmt):
    """The full plain_outlier workload with TKQ_Q_RECIPROCAL, through the tensor
    API (use_sf_inv): codes and scales bit-exact against the oracle's
    reciprocal reading, and some codes differ from the quotient reading."""
    x = synth.workload("plain_outlier")["x"]
    xd = to_dev_bf16(x, cuda_device)
    q, s = tkq.per_token_cast(xd, fmt, use_sf_inv=True)
    ro, rs = oracle.per_token_cast_ex(x, fmt, 128, oracle.Q_RECIPROCAL, threads=THREADS)
    parity.assert_bit_exact("codes", q.view(torch.uint8).cpu().numpy(), ro)
    parity.assert_bit_exact("scales", s.cpu().numpy(), rs)
    q2, _ = tkq.per_token_cast(xd, fmt)
    assert not torch.equal(q.view(torch.uint8), q2.view(torch.uint8))


def _pow2_boundary(s0: np.ndarray, tol=2e-6) -> np.ndarray:
    """Groups whose plain scale lies within tol (relative) of a power of two:
    a few ulp of SwiGLU error can move their rounded-up scale by one binade."""
    m, _ = np.frexp(s0.astype(np.float64))
    return (np.abs(m - 0.5) < tol) | (np.abs(m - 1.0) < tol)


@pytest.mark.parametrize("kind", ["swiglu", "backward"])
@pytest.mark.parametrize("flags", [1, 2, 4, 6, 8])
def test_swiglu_sf_layouts(cuda_device, swiglu_kernel, kind, flags):
    if kind == "swiglu":
        d = synth.workload("swiglu_moe", rows=1031)
        x = np.ascontiguousarray(d["x"][:, np.r_[0:896, 2048:2944]])
        out, raw, G = run_ex("swiglu", x, flags, "e4m3", cuda_device, w=d["w"])
        y = oracle.swiglu_values(x, d["w"], threads=THREADS)
    else:
        d = synth.workload("swiglu_bwd", rows=1031)
        x = np.ascontiguousarray(d["x"][:, np.r_[0:384, 2048:2432]])
        dy = np.ascontiguousarray(d["dy"][:, :384])
        out, raw, G = run_ex("backward", x, flags, "e4m3", cuda_device, w=d["w"], dy_bits=dy)
        y = oracle.swiglu_backward_values(x, dy, d["w"], threads=THREADS)
    T = x.shape[0]
    ro, rs = oracle.cast_rows_f32_ex(y, "e4m3", 128, flags, threads=THREADS)
    got = sf_rowmajor(raw, T, G, flags)
    exp = sf_rowmajor(rs.view(np.uint8).ravel(), T, G, flags)
    if flags & 4:  # padding rows of column-major layouts are zero
        T4 = (T + 3) // 4 * 4
        if flags & 2:
            pad = raw.view(np.uint32).reshape(-1, T4)[:, T:]
        else:
            pad = raw.view(np.float32).reshape(G, T4)[:, T:]
        assert np.all(pad == 0)
    _, s0 = oracle.cast_rows_f32(y, "e4m3")
    skip = _pow2_boundary(s0) if flags & 3 else np.zeros_like(s0, bool)
    assert skip.sum() <= 2, "too many groups at a power-of-two boundary"
    keep = ~skip
    parity.assert_scales_close("scales", got[keep], exp[keep])
    ok_rows = np.repeat(keep, 128, axis=1)
    parity.assert_codes_close("codes", out[ok_rows], ro[ok_rows],
                              max_frac=max(1e-4, 1.0 / out.size))


# ---------------------------------------------------------------------------
# ABI behaviour on a GPU
# ---------------------------------------------------------------------------

def test_argument_errors_launch_nothing(cuda_device):
    dev = cuda_device
    x = to_dev_bf16(synth.workload("plain_small", rows=256)["x"], dev)
    out = Guarded(256 * 4096, dev)
    sf = Guarded(256 * 32 * 4, dev)
    xp = ctypes.c_void_p(x.data_ptr())
    s = stream_of(dev)
    cases = [
        (tkq.tkq_per_token_cast(None, out.ptr, sf.ptr, 256, 4096, 128, 0, s), 1),
        (tkq.tkq_per_token_cast(xp, out.ptr, sf.ptr, 256, 4000, 128, 0, s), 2),
        (tkq.tkq_per_token_cast(xp, out.ptr, sf.ptr, -1, 4096, 128, 0, s), 2),
        (tkq.tkq_per_token_cast(xp, out.ptr, sf.ptr, 256, 4096, 64, 0, s), 3),
        (tkq.tkq_per_token_cast(xp, out.ptr, sf.ptr, 256, 4096, 128, 7, s), 4),
        (tkq.tkq_per_token_cast(ctypes.c_void_p(x.data_ptr() + 2), out.ptr, sf.ptr, 256, 4096,
                                128, 0, s), 5),
        (tkq.tkq_per_token_cast(xp, ctypes.c_void_p(x.data_ptr() + 1024), sf.ptr, 256, 4096,
                                128, 0, s), 8),   # TKQ_ERR_ALIAS
        (tkq.tkq_swiglu_cast_t(xp, None, out.ptr, sf.ptr, out.ptr, sf.ptr, 100, 2048, 128, 0, s), 2),
    ]
    for got, exp in cases:
        assert got == exp, (got, exp)
    torch.cuda.synchronize()
    assert np.all(out.buf.cpu().numpy() == GUARD_BYTE)
    assert np.all(sf.buf.cpu().numpy() == GUARD_BYTE)
    # empty batch: OK, nothing launched, NULL pointers accepted
    assert tkq.tkq_per_token_cast(None, None, None, 0, 4096, 128, 0, s) == 0
    assert tkq.tkq_swiglu_cast_t(None, None, None, None, None, None, 0, 2048, 128, 0, s) == 0


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    """A kernel waits on a barrier nothing arrives on: its wait gives up after
    2 ms, the device status word reports the timeout, and the context keeps
    working (a cast afterwards is still correct)."""
    tkq.tkq_read_device_status(clear=True)
    assert tkq.tkq_selftest_wait_timeout(2_000_000, stream_of(cuda_device)) == 0
    assert tkq.tkq_read_device_status() & tkq.DEVICE_TIMEOUT
    # the C call reports it as TKQ_ERR_TIMEOUT (7), with the word in *flags
    import ctypes
    word = ctypes.c_uint32(0)
    assert tkq.load_library().tkq_read_device_status(ctypes.byref(word), 1) == tkq.ERR_TIMEOUT
    assert word.value & tkq.DEVICE_TIMEOUT
    assert tkq.load_library().tkq_read_device_status(ctypes.byref(word), 0) == 0
    assert tkq.tkq_read_device_status() == 0
    x = synth.workload("swiglu", rows=256)["x"]
    out, sf, out_t, sf_t = run_swiglu(x, None, "e4m3", cuda_device, transposed=True)
    ro, rs, rot, rst = oracle.swiglu_cast_t(x, None, "e4m3")
    parity.assert_codes_close("column codes", out_t, rot, max_frac=max(1e-4, 1.0 / out_t.size))
    assert tkq.tkq_read_device_status() == 0


def test_repeated_launches_are_identical(cuda_device):
    """Many launches on the same input: every plain-cast result equals the
    oracle bit for bit and every transposed-cast result equals the first one.
    A shared-memory stage of the transposed cast's ring released to the TMA
    producer before its readers are done shows up here as a rare corrupted
    group."""
    dev = cuda_device
    x = synth.workload("plain_outlier")["x"]
    xd = to_dev_bf16(x, dev)
    ro, rs = oracle.per_token_cast(x, "e4m3", threads=THREADS)
    for _ in range(40):
        out, sf = tkq.per_token_cast(xd, "e4m3")
        torch.cuda.synchronize()
        parity.assert_bit_exact("scales", sf.cpu().numpy(), rs)
        parity.assert_bit_exact("codes", out.view(torch.uint8).cpu().numpy(), ro)
    xs = to_dev_bf16(synth.workload("swiglu_t", rows=16384)["x"], dev)
    ref = [t.clone() for t in tkq.swiglu_forward_and_per_token_cast(xs, with_transpose=True)]
    for _ in range(40):
        cur = tkq.swiglu_forward_and_per_token_cast(xs, with_transpose=True)
        torch.cuda.synchronize()
        for a, b in zip(ref, cur):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert tkq.tkq_read_device_status() == 0


def test_runs_on_caller_stream(cuda_device):
    dev = cuda_device
    x = synth.workload("plain_small")["x"]
    xd = to_dev_bf16(x, dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        out, sf = tkq.per_token_cast(xd, "e4m3")
    side.synchronize()
    ro, rs = oracle.per_token_cast(x, "e4m3", threads=THREADS)
    parity.assert_bit_exact("codes", out.view(torch.uint8).cpu().numpy(), ro)
    parity.assert_bit_exact("scales", sf.cpu().numpy(), rs)


def test_tensor_api_shapes_and_dtypes(cuda_device):
    dev = cuda_device
    x = to_dev_bf16(synth.workload("swiglu", rows=256)["x"], dev)
    out, sf, out_t, sf_t = tkq.swiglu_forward_and_per_token_cast(x, "e5m2", with_transpose=True)
    assert out.dtype == torch.float8_e5m2 and out.shape == (256, 2048)
    assert sf.shape == (256, 16) and out_t.shape == (2048, 256) and sf_t.shape == (2048, 2)
    with pytest.raises(tkq.TkqError):
        tkq.swiglu_forward_and_per_token_cast(x[:100].contiguous(), with_transpose=True)
