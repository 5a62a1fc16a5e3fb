"""Ordering of consecutive casts on one stream.

The casts are launched with programmatic dependent launch allowed, so a cast's
CTAs may be scheduled while the kernel before it is still draining; each cast
waits at entry (griddepcontrol.wait) until that kernel has completed and its
memory is visible.  These tests chain casts with no synchronization between
them, through read-after-write (a cast reads what the previous one wrote) and
write-after-read (a cast overwrites what the previous one read) hazards, many
times over, on a stream and inside a CUDA graph, and require the bytes of a
chain run with a full device synchronization after every launch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import fp8_activation_quantization_gb300 as tkq
from fp8_activation_quantization_gb300 import synth
from tests.test_gpu_parity import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    tkq.load_library()
    yield


def _chain(x0, rounds, sync):
    """rounds x: codes, sf = per_token_cast(x); x = cast_back(codes, sf) as bf16
    written into x itself (the buffer the previous cast read), then the
    SwiGLU cast and its transposed copy of [x | x].  Returns every output."""
    x = x0.clone()
    outs = []
    for _ in range(rounds):
        q, s = tkq.per_token_cast(x, "e4m3")               # reads x
        if sync:
            torch.cuda.synchronize()
        tkq.cast_back(q.view(torch.uint8), s, fmt="e4m3", group_size=(1, 128),
                      out_dtype=torch.bfloat16, out=x)       # reads q, s; writes x
        if sync:
            torch.cuda.synchronize()
        xx = torch.cat([x, x], dim=1)
        q2, s2, qt, st = tkq.swiglu_forward_and_per_token_cast(xx, with_transpose=True)
        if sync:
            torch.cuda.synchronize()
        outs += [q.view(torch.uint8).clone(), s.clone(), q2.view(torch.uint8).clone(), s2.clone(),
                 qt.view(torch.uint8).clone(), st.clone()]
    outs.append(x.clone())
    return outs


def _same(a, b):
    assert len(a) == len(b)
    for i, (u, v) in enumerate(zip(a, b)):
        assert torch.equal(u.view(torch.uint8), v.view(torch.uint8)), f"output {i} differs"


def test_chained_casts_equal_synchronized_chain(cuda_device):
    x0 = to_dev_bf16(synth.outlier_bf16(91, 1, 1024, 1024, zero_row_every=0), cuda_device)
    ref = _chain(x0, 6, sync=True)
    for _ in range(20):
        got = _chain(x0, 6, sync=False)
        torch.cuda.synchronize()
        _same(got, ref)
    assert tkq.tkq_read_device_status() == 0


def test_chained_casts_in_a_graph_equal_synchronized_chain(cuda_device):
    x0 = to_dev_bf16(synth.outlier_bf16(92, 1, 512, 768, zero_row_every=0), cuda_device)
    ref = _chain(x0, 4, sync=True)
    x = x0.clone()
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _chain(x, 4, sync=False)        # first calls outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        got = _chain(x, 4, sync=False)
    for _ in range(10):
        x.copy_(x0)          # the chain rewrites x; it starts from x0 each time
        g.replay()
        torch.cuda.synchronize()
        # the chain clones x0 into its own buffer, so replays do not depend on x
        _same(got, ref)
    assert tkq.tkq_read_device_status() == 0


def test_writes_after_reads_on_one_buffer(cuda_device):
    """A cast back that overwrites the very input of the cast before it, again
    and again: every round's codes must be those of the value the buffer held
    when that round's cast was issued."""
    x0 = to_dev_bf16(synth.outlier_bf16(93, 1, 2048, 4096, zero_row_every=0), cuda_device)
    x = x0.clone()
    rounds = 8
    got = []
    for _ in range(rounds):
        q, s = tkq.per_token_cast(x)
        tkq.cast_back(q.view(torch.uint8), s, fmt="e4m3", group_size=(1, 128),
                      out_dtype=torch.bfloat16, out=x)
        got.append(q.view(torch.uint8))
    torch.cuda.synchronize()
    y = x0.clone()
    for r in range(rounds):
        q, s = tkq.per_token_cast(y)
        torch.cuda.synchronize()
        assert torch.equal(q.view(torch.uint8), got[r]), f"round {r}"
        tkq.cast_back(q.view(torch.uint8), s, fmt="e4m3", group_size=(1, 128),
                      out_dtype=torch.bfloat16, out=y)
        torch.cuda.synchronize()
    assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_short_output_buffers_are_refused_before_launch(cuda_device):
    """A caller-supplied output smaller than what the call writes raises before
    anything is launched: the buffer around it keeps its bytes."""
    x = to_dev_bf16(synth.outlier_bf16(94, 1, 256, 1024, zero_row_every=0), cuda_device)
    guard = torch.full((256 * 1024 + 4096,), 0xA5, dtype=torch.uint8, device=cuda_device)
    short = guard[:256 * 1024 - 16]
    with pytest.raises(ValueError):
        tkq.per_token_cast(x, out=short)
    sf = torch.empty(256, 8, dtype=torch.float32, device=cuda_device)
    with pytest.raises(ValueError):
        tkq.per_token_cast(x, out=guard[:256 * 1024], out_sf=sf[:255])
    xx = torch.cat([x, x], dim=1)
    with pytest.raises(ValueError):
        tkq.swiglu_forward_and_per_token_cast(xx, with_transpose=True,
                                              out_t=guard[:1024 * 255])
    q, s = tkq.per_token_cast(x)
    with pytest.raises(TypeError):
        tkq.cast_back(q, s, out_dtype=torch.bfloat16,
                      out=torch.empty(256, 1024, dtype=torch.float32, device=cuda_device))
    torch.cuda.synchronize()
    assert torch.all(guard == 0xA5)


def _chain_tiles(x0, w, rounds, sync):
    """The tile, ring and backward casts chained the same way: per-channel
    (transposed) -> cast back -> per-block -> cast back into the per-block
    cast's own input -> SwiGLU cast (x weight) of that -> cast back -> SwiGLU
    backward cast, then the in-place per-channel cast of x and its cast back
    into x for the next round."""
    x = x0.clone()
    outs = []

    def step():
        if sync:
            torch.cuda.synchronize()

    for _ in range(rounds):
        qt, st = tkq.per_channel_cast(x, transpose=True)            # reads x
        step()
        yt = tkq.cast_back(qt.view(torch.uint8), st, fmt="e4m3", group_size=(1, 128),
                           out_dtype=torch.bfloat16)
        step()
        qb, sb = tkq.per_block_cast(yt)                              # reads yt
        step()
        tkq.cast_back(qb.view(torch.uint8), sb, fmt="e4m3", group_size=(128, 128),
                      out_dtype=torch.bfloat16, out=yt)              # writes yt
        step()
        q2, s2 = tkq.swiglu_forward_and_per_token_cast(yt, topk_weights=w)
        step()
        dy = tkq.cast_back(q2.view(torch.uint8), s2, fmt="e4m3", group_size=(1, 128),
                           out_dtype=torch.bfloat16)
        step()
        q3, s3 = tkq.swiglu_backward_and_per_token_cast(yt, dy, topk_weights=w)
        step()
        qc, sc = tkq.per_channel_cast(x)                             # reads x
        step()
        tkq.cast_back(qc.view(torch.uint8), sc, fmt="e4m3", group_size=(128, 1),
                      out_dtype=torch.bfloat16, out=x)               # writes x
        step()
        outs += [t.view(torch.uint8).clone() if t.element_size() == 1 else t.clone()
                 for t in (qt, st, qb, sb, q2, s2, q3, s3, qc, sc)]
    outs.append(x.clone())
    return outs


def test_chained_tile_ring_and_backward_casts(cuda_device, swiglu_kernel):
    """Every other cast in one unsynchronized chain, through both SwiGLU forward
    kernels, against the same chain with a synchronization after each launch."""
    x0 = to_dev_bf16(synth.outlier_bf16(95, 1, 512, 768, zero_row_every=0), cuda_device)
    w = torch.rand(768, generator=torch.Generator().manual_seed(96)).to(cuda_device)
    ref = _chain_tiles(x0, w, 3, sync=True)
    for _ in range(10):
        got = _chain_tiles(x0, w, 3, sync=False)
        torch.cuda.synchronize()
        _same(got, ref)
    assert tkq.tkq_read_device_status() == 0
