"""Multi-rank orchestration of bench.py (CPU, no GPU).

The benchmark scales weakly: with N ranks the batch holds N workloads' worth of
rows, and shard_rows gives each rank one contiguous range of it.  These tests
check that the ranges tile the batch, that a rank's inputs are exactly its rows
of the one seeded batch, that two gloo ranks quantizing their shards reproduce
the whole batch quantized at once (the oracle on both sides), that the timing
reduction is the slowest rank's time, that `--gpus 2` fails loudly where two
GPUs are not visible, and that the reference arm under two ranks runs on rank 0
alone and prints one line.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from fp8_activation_quantization_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", sorted(bench.KERNEL_OF))
@pytest.mark.parametrize("ws", [1, 2, 3, 8])
def test_rank_shards_tile_the_global_batch(workload, ws):
    T = synth.WORKLOADS[bench.SYNTH_OF.get(workload, workload)][0]
    spans = [bench.rank_shard(workload, ws, r) for r in range(ws)]
    assert all(g == T * ws for _, _, g in spans)
    assert spans[0][0] == 0 and spans[-1][1] == T * ws
    for (a, b, _), (c, d, _) in zip(spans, spans[1:]):
        assert b == c
    # weak scaling: every rank holds one workload's rows
    assert all(b - a == T for a, b, _ in spans)
    if T % 128 == 0:
        assert all(a % 128 == 0 for a, _, _ in spans)


@pytest.mark.parametrize("workload", ["plain_outlier", "swiglu_moe", "swiglu_bwd", "cast_back",
                                      "per_block"])
def test_rank_inputs_are_rows_of_one_batch(workload):
    syn = bench.SYNTH_OF.get(workload, workload)
    rows = 1000   # not a multiple of the generator's chunk
    whole = synth.workload(syn, rows=3 * rows)
    for r in range(3):
        a, b, g = bench.rank_shard(workload, 3, r, rows=rows)
        assert (b - a, g) == (rows, 3 * rows)
        part = synth.workload(syn, rows=b - a, row_begin=a)
        assert part.keys() == whole.keys()
        for k in whole:
            assert np.array_equal(part[k], whole[k][a:b]), (workload, r, k)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROWS_PER_RANK = 256


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        a, b, g = bench.rank_shard("swiglu_t", world, rank, rows=ROWS_PER_RANK)
        d = synth.workload("swiglu_t", rows=b - a, row_begin=a)
        res = oracle.swiglu_cast_t(d["x"], None)
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, a, b, res))
        slowest = bench.max_over_ranks(0.5 + rank, world)
        if rank == 0:
            spans = [(r, a_, b_) for r, a_, b_, _ in gathered]
            full = oracle.swiglu_cast_t(synth.workload("swiglu_t", rows=g)["x"], None)
            parts = [x[3] for x in sorted(gathered)]
            ok = spans == [(r, r * ROWS_PER_RANK, (r + 1) * ROWS_PER_RANK) for r in range(world)]
            ok &= np.array_equal(np.concatenate([p[0] for p in parts]), full[0])
            ok &= np.array_equal(np.concatenate([p[1] for p in parts]), full[1])
            ok &= np.array_equal(np.concatenate([p[2] for p in parts], axis=1), full[2])
            ok &= np.array_equal(np.concatenate([p[3] for p in parts], axis=1), full[3])
            ok &= slowest == 0.5 + world - 1
            q.put(bool(ok))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_quantize_their_shards_of_one_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) is True


def _bench(*args, timeout=300):
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def test_more_gpus_than_visible_fails_loudly():
    have = torch.cuda.device_count()
    r = _bench("--gpus", str(have + 1), "--steps", "1", "--warmup", "3", "--no-extras")
    assert r.returncode != 0
    assert f"needs {have + 1} GPUs" in r.stderr
    assert not r.stdout.strip()


def test_reference_arm_under_two_ranks_prints_one_line():
    r = _bench("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
               "--workload", "plain_small", "--ref-seconds", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["config"] == bench.workload_config("plain_small", "e4m3", 2)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
