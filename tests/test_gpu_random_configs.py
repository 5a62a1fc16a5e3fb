"""Randomized configurations of every entry point against the oracle (seeded):
shapes with ragged row counts, both formats, every scale layout, with and
without routing weights and clamp.  Exact ops are compared bit for bit, the
SwiGLU ops with the SwiGLU tolerance; plus a multi-threaded run in which four
host threads launch on their own streams at once."""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import pytest
import torch

import oracle
import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests import parity
from tests.test_gpu_parity import to_dev_bf16

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))
FLAGS = [0, 1, 2, 4, 5, 6, 7, 8, 12, 15]


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def _opts(flags):
    return dict(round_sf=bool(flags & 1), use_packed_ue8m0=bool(flags & 2),
                use_tma_aligned_col_major_sf=bool(flags & 4), use_sf_inv=bool(flags & 8))


def _raw(t):
    return np.ascontiguousarray(t.contiguous().view(torch.uint8).cpu().numpy()).ravel()


@pytest.mark.parametrize("case", range(24))
def test_random_row_casts(cuda_device, case):
    rng = np.random.default_rng(1000 + case)
    T = int(rng.choice([1, 3, 31, 32, 33, 127, 500, 1029]))
    C = 128 * int(rng.integers(1, 12))
    fmt = str(rng.choice(["e4m3", "e5m2"]))
    flags = int(rng.choice(FLAGS))
    kind = str(rng.choice(["bf16", "f32"]))
    dev = cuda_device
    if kind == "bf16":
        x = synth.outlier_bf16(case, 7, T, C, zero_row_every=int(rng.choice([0, 5])))
        q, s = tkq.per_token_cast(to_dev_bf16(x, dev), fmt, **_opts(flags))
        y = synth.bf16_bits_to_f32(x)
    else:
        y = (rng.standard_normal((T, C)) * np.exp2(rng.uniform(-30, 30, (T, 1)))).astype(np.float32)
        q, s = tkq.per_token_cast(torch.from_numpy(y).to(dev), fmt, **_opts(flags))
    e_q, e_s = oracle.cast_rows_f32_ex(y, fmt, flags=flags)
    parity.assert_bit_exact("codes", q.view(torch.uint8).cpu().numpy(), e_q)
    parity.assert_bit_exact("scales", _raw(s), np.ascontiguousarray(e_s).view(np.uint8).ravel())


@pytest.mark.parametrize("case", range(16))
def test_random_swiglu_casts(cuda_device, swiglu_kernel, case):
    rng = np.random.default_rng(2000 + case)
    transposed = bool(case % 4 == 0)
    T = 128 * int(rng.integers(1, 6)) if transposed else int(rng.choice([1, 7, 64, 129, 700]))
    H = 128 * int(rng.integers(1, 6))
    fmt = str(rng.choice(["e4m3", "e5m2"]))
    weighted = bool(rng.integers(0, 2))
    clamp = float(rng.choice([0.75, 2.5])) if rng.integers(0, 2) else None
    dev = cuda_device
    x = synth.swiglu_bf16(case, 11, T, H, gate_std=float(rng.choice([1.0, 2.0])))
    w = synth.routing_weights(case, 12, -(-T // 8))[:T] if weighted else None
    xd = to_dev_bf16(x, dev)
    wd = None if w is None else torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev) if clamp is not None else None
    kw = dict(topk_weights=wd, use_clamp=clamp is not None, swiglu_clamp_value=clamp,
              clamp_count=cnt)
    if clamp is None:
        y = oracle.swiglu_values(x, w)
        n_exp = None
    else:
        y, n_exp = oracle.swiglu_values(x, w, clamp=clamp)
    e_q, e_s = oracle.cast_rows_f32(y, fmt)
    q_ref = y / np.repeat(e_s, 128, axis=1)
    if transposed:
        q, s, qt, st = tkq.swiglu_forward_and_per_token_cast(xd, fmt, with_transpose=True, **kw)
        e_qt, e_st = oracle.cast_cols_f32(y, fmt)
        parity.assert_scales_close("sf_t", st.cpu().numpy(), e_st)
        parity.assert_codes_differ_only_at_ties("codes_t", qt.view(torch.uint8).cpu().numpy(), e_qt,
                                                y.T / np.repeat(e_st, 128, axis=1), fmt)
    else:
        q, s = tkq.swiglu_forward_and_per_token_cast(xd, fmt, **kw)
    parity.assert_scales_close("sf", s.cpu().numpy(), e_s)
    parity.assert_codes_differ_only_at_ties("codes", q.view(torch.uint8).cpu().numpy(), e_q, q_ref,
                                            fmt)
    if clamp is not None:
        assert int(cnt.item()) == n_exp


@pytest.mark.parametrize("case", range(12))
def test_random_tile_casts_and_cast_back(cuda_device, case):
    rng = np.random.default_rng(3000 + case)
    T = int(rng.choice([1, 100, 128, 255, 640]))
    C = 128 * int(rng.integers(1, 9))
    fmt = str(rng.choice(["e4m3", "e5m2"]))
    dev = cuda_device
    x = synth.outlier_bf16(case, 13, T, C, zero_row_every=0)
    xd = to_dev_bf16(x, dev)
    q, s = tkq.per_block_cast(xd, fmt)
    e_q, e_s = oracle.per_block_cast(x, fmt)
    parity.assert_bit_exact("block codes", q.view(torch.uint8).cpu().numpy(), e_q)
    parity.assert_bit_exact("block scales", s.cpu().numpy(), e_s)
    out_dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
    yb = tkq.cast_back(q, s, group_size=(128, 128), out_dtype=out_dtype)
    ey = torch.from_numpy(oracle.cast_back(e_q, e_s, 128, 128, fmt)).to(out_dtype)
    assert torch.equal(yb.cpu().view(torch.uint8), ey.view(torch.uint8))
    if T % 128 == 0:
        tr = bool(rng.integers(0, 2))
        q, s = tkq.per_channel_cast(xd, fmt, transpose=tr)
        e_q, e_s = oracle.per_channel_cast(x, fmt, transpose=tr)
        parity.assert_bit_exact("channel codes", q.view(torch.uint8).cpu().numpy(), e_q)
        parity.assert_bit_exact("channel scales", s.cpu().numpy(), e_s)


def test_concurrent_host_threads(cuda_device):
    """Four host threads, each on its own stream, run the row, SwiGLU, tile and
    cast-back kernels 20 times each at once; every result equals the same call
    made alone."""
    dev = cuda_device
    xs = [to_dev_bf16(synth.outlier_bf16(k, 21, 384, 768), dev) for k in range(4)]
    sw = [to_dev_bf16(synth.swiglu_bf16(k, 22, 256, 256), dev) for k in range(4)]

    def work(k):
        return [tkq.per_token_cast(xs[k]), tkq.swiglu_forward_and_per_token_cast(sw[k], with_transpose=True),
                tkq.per_block_cast(xs[k]), tkq.per_channel_cast(xs[k], transpose=True)]

    ref = [work(k) for k in range(4)]
    torch.cuda.synchronize()
    errors = []

    def run(k):
        try:
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                for _ in range(20):
                    got = work(k)
                s.synchronize()
            for a, b in zip(got, ref[k]):
                for ta, tb in zip(a, b):
                    if not torch.equal(ta.view(torch.uint8), tb.view(torch.uint8)):
                        errors.append(f"thread {k}: output differs")
        except Exception as e:  # surfaced below
            errors.append(f"thread {k}: {e!r}")

    threads = [threading.Thread(target=run, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert tkq.tkq_read_device_status() == 0


@pytest.mark.parametrize("sms", ["1", "3"])
def test_tiny_persistent_grids_give_the_same_bytes(cuda_device, sms, monkeypatch):
    """With the grid capped at a few SMs (TKQ_NUM_SMS), every persistent CTA
    walks many tiles and its copy ring wraps many times; results must equal
    the full-grid results byte for byte."""
    dev = cuda_device
    x = to_dev_bf16(synth.outlier_bf16(31, 1, 1000, 1024, zero_row_every=0), dev)
    xs = to_dev_bf16(synth.swiglu_bf16(32, 2, 1024, 512, gate_std=2.0), dev)
    codes = torch.from_numpy(synth.random_bytes(33, 3, 1000, 1024)).to(dev)
    sfc = torch.from_numpy(synth.log_uniform_f32(34, 4, (1000, 8), -10.0, 2.0)).to(dev)

    def run():
        return [*tkq.per_token_cast(x), *tkq.swiglu_forward_and_per_token_cast(xs, with_transpose=True),
                *tkq.swiglu_backward_and_per_token_cast(xs, xs[:, :512].contiguous()),
                *tkq.per_block_cast(x), *tkq.per_channel_cast(xs, transpose=True),
                tkq.cast_back(codes, sfc, fmt="e4m3", out_dtype=torch.bfloat16)]

    ref = run()
    torch.cuda.synchronize()
    monkeypatch.setenv("TKQ_NUM_SMS", sms)
    got = run()
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"output {i} differs"
    assert tkq.tkq_read_device_status() == 0
