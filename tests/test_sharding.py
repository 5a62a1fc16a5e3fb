"""Row sharding across ranks (host logic, CPU only).

Two gloo ranks each quantize their shard of a batch with the CPU oracle; the
gathered shards must equal the whole batch quantized at once, which is what
makes the multi-GPU path exchange-free.  The timing reduction used by the
benchmark (max over ranks) is checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_activation_quantization_gb300.sharding import shard_rows


@pytest.mark.parametrize("T,world,align", [(0, 2, 1), (1, 2, 1), (1031, 3, 1), (1024, 4, 128),
                                           (128 * 7, 2, 128), (128 * 3, 8, 128)])
def test_shards_partition_the_rows(T, world, align):
    spans = [shard_rows(T, world, r, align) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == T
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c
    sizes = [b - a for a, b in spans]
    assert all(s % align == 0 for s in sizes)
    assert max(sizes) - min(sizes) <= align


def test_bad_arguments():
    with pytest.raises(ValueError):
        shard_rows(100, 2, 0, 128)
    with pytest.raises(ValueError):
        shard_rows(128, 2, 2, 128)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from fp8_activation_quantization_gb300 import synth
        d = synth.workload("swiglu_moe", rows=512)
        x = np.ascontiguousarray(d["x"][:, np.r_[0:256, 2048:2304]])
        w = d["w"]
        a, b = shard_rows(x.shape[0], world, rank, 128)
        out, sf, out_t, sf_t = oracle.swiglu_cast_t(np.ascontiguousarray(x[a:b]), w[a:b])
        gathered = [None] * world
        dist.all_gather_object(gathered, (a, b, out, sf, out_t, sf_t))
        t = torch.tensor([0.25 * (rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            full = oracle.swiglu_cast_t(x, w)
            out_g = np.concatenate([g[2] for g in gathered])
            sf_g = np.concatenate([g[3] for g in gathered])
            out_t_g = np.concatenate([g[4] for g in gathered], axis=1)
            sf_t_g = np.concatenate([g[5] for g in gathered], axis=1)
            ok = (np.array_equal(out_g, full[0]) and np.array_equal(sf_g, full[1])
                  and np.array_equal(out_t_g, full[2]) and np.array_equal(sf_t_g, full[3])
                  and abs(float(t.item()) - 0.25 * world) < 1e-12)
            q.put(bool(ok))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_shards_match_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world = 2
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) is True
