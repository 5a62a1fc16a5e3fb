"""The access-checked build (libtkq_checked.so, -DTKQ_CHECKED), the stand-in
for a memory checker: every global load and store of the kernels is checked
against the buffers of the call before it is made.

1. Every entry point, on ragged and multi-tile shapes and with every option,
   runs in the checked build without a single refused access, and gives the
   same bytes as the release build.
2. The checks themselves: with TKQ_CHECK_WITHHOLD=16 the last 16 bytes of
   every output are left out of the checked table (the buffers are still
   allocated, so no access leaves memory the call owns), and every entry
   point must report a refused store whose address lies in one of those
   withheld tails.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests.test_gpu_parity import to_dev_bf16

pytestmark = pytest.mark.gpu

WITHHOLD = 16


@pytest.fixture(scope="module", autouse=True)
def _libraries(cuda_device):
    import __graft_entry__
    from fp8_activation_quantization_gb300 import _build
    __graft_entry__.build()
    _build.build(checked=True)
    tkq.load_library()
    assert not tkq.tkq_checked_build()
    with tkq.use_checked_library():
        assert tkq.tkq_checked_build()
    yield


def _dev_f32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)


def _cases(dev):
    """(name, fn) pairs; fn() launches one call and returns its output tensors
    (inputs are made once, outside fn)."""
    cases = []
    for T, C, flags in [(1, 128, 0), (7, 384, 6), (129, 896, 7), (1031, 256, 8), (5, 640, 5)]:
        x = to_dev_bf16(synth.outlier_bf16(T, C, T, C, zero_row_every=3), dev)
        opts = dict(round_sf=bool(flags & 1), use_packed_ue8m0=bool(flags & 2),
                    use_tma_aligned_col_major_sf=bool(flags & 4), use_sf_inv=bool(flags & 8))
        cases.append((f"per_token bf16 {T}x{C} flags {flags}",
                      lambda x=x, o=opts: tkq.per_token_cast(x, "e4m3", **o)))
    for T, C, flags in [(3, 256, 0), (130, 384, 4)]:
        xf = _dev_f32(np.random.default_rng(T).standard_normal((T, C)), dev)
        cases.append((f"per_token fp32 {T}x{C} flags {flags}",
                      lambda x=xf, f=flags: tkq.per_token_cast(
                          x, "e5m2", use_tma_aligned_col_major_sf=bool(f & 4))))
    for T, H, weighted, clamp, flags in [(1, 128, False, None, 0), (129, 384, True, None, 6),
                                         (33, 256, True, 2.0, 0), (70, 128, False, 0.7, 4)]:
        x = to_dev_bf16(synth.swiglu_bf16(T, H, T, H, gate_std=2.0), dev)
        w = _dev_f32(synth.routing_weights(T, 3, -(-T // 8))[:T], dev) if weighted else None
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        kw = dict(topk_weights=w, use_tma_aligned_col_major_sf=bool(flags & 4),
                  use_packed_ue8m0=bool(flags & 2))
        if clamp is not None:
            kw.update(use_clamp=True, swiglu_clamp_value=clamp, clamp_count=cnt)

        def fn(x=x, kw=kw, cnt=cnt):
            cnt.zero_()
            return (*tkq.swiglu_forward_and_per_token_cast(x, **kw), cnt)
        cases.append((f"swiglu {T}x{H} w={weighted} clamp={clamp} flags {flags}", fn))
    for T, H, weighted, clamp in [(128, 128, False, None), (256, 384, True, None),
                                  (384, 256, True, 4.0), (128, 256, False, 1.3)]:
        x = to_dev_bf16(synth.swiglu_bf16(T + 1, H, T, H, gate_std=2.0), dev)
        w = _dev_f32(synth.routing_weights(T, 4, T // 8), dev) if weighted else None
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        kw = dict(topk_weights=w, with_transpose=True,
                  use_packed_ue8m0=bool(T == 384), use_tma_aligned_col_major_sf=bool(T >= 256))
        if clamp is not None:
            kw.update(use_clamp=True, swiglu_clamp_value=clamp, clamp_count=cnt)

        def fn(x=x, kw=kw, cnt=cnt):
            cnt.zero_()
            return (*tkq.swiglu_forward_and_per_token_cast(x, **kw), cnt)
        cases.append((f"swiglu_t {T}x{H} w={weighted} clamp={clamp}", fn))
    for T, H, weighted in [(7, 128, False), (129, 256, True)]:
        x = to_dev_bf16(synth.swiglu_bf16(T + 2, H, T, H), dev)
        dy = to_dev_bf16(synth.normal_bf16(T + 3, H, T, H), dev)
        w = _dev_f32(synth.routing_weights(T, 5, -(-T // 8))[:T], dev) if weighted else None
        cases.append((f"swiglu backward {T}x{H} w={weighted}",
                      lambda x=x, dy=dy, w=w: tkq.swiglu_backward_and_per_token_cast(
                          x, dy, topk_weights=w)))
    for T, C in [(128, 128), (256, 384)]:
        x = to_dev_bf16(synth.outlier_bf16(T + 4, C, T, C, zero_row_every=0), dev)
        for tr in (False, True):
            cases.append((f"per_channel {T}x{C} transpose={tr}",
                          lambda x=x, tr=tr: tkq.per_channel_cast(x, transpose=tr)))
    for T, C in [(1, 128), (129, 384), (300, 256)]:
        x = to_dev_bf16(synth.outlier_bf16(T + 5, C, T, C, zero_row_every=0), dev)
        cases.append((f"per_block {T}x{C}", lambda x=x: tkq.per_block_cast(x)))
    for T, C, group in [(1, 128, (1, 128)), (129, 384, (1, 128)), (256, 256, (128, 1)),
                        (300, 384, (128, 128))]:
        codes = torch.from_numpy(synth.random_bytes(T, C, T, C)).to(dev)
        gr, gc = group
        sf = _dev_f32(synth.log_uniform_f32(T, C, (-(-T // gr), C // gc), -8.0, 2.0), dev)
        for dt in (torch.float32, torch.bfloat16):
            cases.append((f"cast_back {T}x{C} groups {group} {dt}",
                          lambda q=codes, s=sf, g=group, dt=dt: (tkq.cast_back(
                              q, s, fmt="e4m3", group_size=g, out_dtype=dt),)))
    for n, fmt in [(4, "e4m3"), (1028, "e5m2")]:
        xv = _dev_f32(np.random.default_rng(n).standard_normal(n) * 300.0, dev)
        cases.append((f"fp8_encode {n} {fmt}", lambda x=xv, f=fmt: (tkq.fp8_encode(x, f),)))
    for T, H, weighted in [(3, 128, False), (129, 256, True)]:
        x = to_dev_bf16(synth.swiglu_bf16(T + 6, H, T, H), dev)
        w = _dev_f32(synth.routing_weights(T, 6, -(-T // 8))[:T], dev) if weighted else None
        cases.append((f"swiglu_values {T}x{H} w={weighted}",
                      lambda x=x, w=w: (tkq.swiglu_values(x, w),)))
    return cases


def _bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def test_every_entry_point_stays_inside_its_buffers(cuda_device, swiglu_kernel):
    tkq.tkq_read_device_status(clear=True)
    for name, fn in _cases(cuda_device):
        ref = [_bytes(t) for t in fn()]
        with tkq.use_checked_library():
            tkq.tkq_read_device_status(clear=True)
            tkq.tkq_read_check_address(clear=True)
            got = [_bytes(t) for t in fn()]
            status = tkq.tkq_read_device_status(clear=True)
            bad = tkq.tkq_read_check_address(clear=True)
        assert status == 0 and bad == 0, f"{name}: status {status}, refused address {bad:#x}"
        for i, (a, b) in enumerate(zip(got, ref)):
            assert np.array_equal(a, b), f"{name}: output {i} differs from the release build"


def test_withheld_output_tails_are_refused_and_reported(cuda_device, swiglu_kernel, monkeypatch):
    monkeypatch.setenv("TKQ_CHECK_WITHHOLD", str(WITHHOLD))
    cases = _cases(cuda_device)
    with tkq.use_checked_library():
        tkq.tkq_read_device_status(clear=True)
        tkq.tkq_read_check_address(clear=True)
        for name, fn in cases:
            outs = fn()
            status = tkq.tkq_read_device_status(clear=True)
            bad = tkq.tkq_read_check_address(clear=True)
            assert status & tkq.DEVICE_OUT_OF_BOUNDS, f"{name}: no refused access reported"
            assert bad >> 63 == 1, f"{name}: the refused access is not a store ({bad:#x})"
            addr = bad & ((1 << 63) - 1)
            tails = [(t.data_ptr() + t.numel() * t.element_size() - min(
                WITHHOLD, t.numel() * t.element_size()), t.data_ptr() + t.numel() * t.element_size())
                for t in outs]
            assert any(lo <= addr < hi for lo, hi in tails), \
                f"{name}: refused address {addr:#x} is not in a withheld tail {tails}"
