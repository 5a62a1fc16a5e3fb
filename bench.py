"""Benchmark of the GB300 per-token FP8 activation quantization path.

One step = one launch of the fused SwiGLU + per-token E4M3 cast + transposed
cast (every step of the path: row-tile load, SwiGLU epilogue, group absmax,
scale, FP8 pack, transposed copy) on the bf16 [131072, 4096] gate|up workload
(H = 2048).  Inputs are resident in HBM when the timed region starts and are
larger than L2 (1.07 GB per step), so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Metric: HBM GB/s of algorithmic bytes (bytes
read + bytes written), with the fraction of the measured HBM peak and rows/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--fmt e4m3|e5m2] [--no-extras]

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores instead: the reference arm of this benchmark.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused SwiGLU+FP8 per-token cast HBM GB/s and % of GB300 peak; rows/sec"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "swiglu_t"

# workload -> (kernel, rows, C or 2H, fmt list)
KERNEL_OF = {
    "plain_small": "per_token_cast",
    "plain_outlier": "per_token_cast",
    "swiglu": "swiglu_cast",
    "swiglu_moe": "swiglu_cast",
    "swiglu_t": "swiglu_cast_t",
    "swiglu_bwd": "swiglu_backward_cast",
    "per_channel": "per_channel_cast",
    "per_channel_t": "per_channel_cast_t",
    "per_block": "per_block_cast",
    "cast_back": "cast_back",
    "swiglu_clamp": "swiglu_cast_clamp",
    "swiglu_t_clamp": "swiglu_cast_t_clamp",
    "plain_f32": "per_token_cast_f32",
}
# bench workload -> seeded input set, where the names differ
SYNTH_OF = {"per_channel_t": "per_channel", "swiglu_clamp": "swiglu",
            "swiglu_t_clamp": "swiglu_t"}
# SwiGLU clamp bound of the clamped workloads (swiglu_clamp: gate ~ N(0, 2^2),
# ~2.3 % of the gates lie above it; swiglu_t_clamp: gate and up ~ N(0, 1), about
# one value in 10^4 is clamped; the clamp runs on every element either way)
CLAMP_VALUE = 4.0
KERNEL_SOURCES = {
    "per_token_cast": ["token_cast.cu", "tkq_device.cuh"],
    "swiglu_cast": ["row_cast.cu", "swiglu_flat.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "swiglu_cast_t": ["swiglu_cast_t.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "swiglu_backward_cast": ["row_cast.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "per_channel_cast": ["tile_cast.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "per_channel_cast_t": ["tile_cast.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "per_block_cast": ["tile_cast.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "cast_back": ["cast_back.cu", "tkq_device.cuh"],
    "swiglu_cast_clamp": ["row_cast.cu", "swiglu_flat.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "swiglu_cast_t_clamp": ["swiglu_cast_t.cu", "tkq_device.cuh", "tkq_async.cuh"],
    "per_token_cast_f32": ["token_cast.cu", "tkq_device.cuh"],
}


def algorithmic_bytes(workload: str, T: int, C: int, weighted: bool) -> int:
    """Bytes the operation must read and write once (per launch)."""
    kern = KERNEL_OF[workload]
    if kern == "per_token_cast":
        return T * C * 2 + T * C + T * (C // 128) * 4
    if kern == "per_token_cast_f32":
        return T * C * 4 + T * C + T * (C // 128) * 4
    if kern in ("per_channel_cast", "per_channel_cast_t"):
        return T * C * 2 + T * C + (T // 128) * C * 4
    if kern == "per_block_cast":
        return T * C * 2 + T * C + -(-T // 128) * (C // 128) * 4
    if kern == "cast_back":
        # read codes and per-token scales, write bf16
        return T * C + T * (C // 128) * 4 + T * C * 2
    H = C // 2
    if kern == "swiglu_backward_cast":
        # read gate|up and dy, write codes and scales of [dg | du]
        return T * 4 * H + T * 2 * H + T * 2 * H + T * (2 * H // 128) * 4 + (T * 4 if weighted else 0)
    b = T * 2 * H * 2 + T * H + T * (H // 128) * 4
    if weighted:
        b += T * 4
    if kern in ("swiglu_cast_t", "swiglu_cast_t_clamp"):
        b += T * H + H * (T // 128) * 4
    return b


def kernel_source_hash(kern: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kern]:
        with open(os.path.join(ROOT, "fp8_activation_quantization_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kern: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel and
    workload, if the summary was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kern}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    s = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash(kern):
        return None
    return int(m.group(1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (measured copy bandwidth)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        base = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                "-lms", "100"]
        for cmd in ([base + ["-i", self.gpu_id]] if self.gpu_id else []) + [base]:
            try:
                self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
                continue
            time.sleep(0.3)
            if self.proc.poll() is None:  # still sampling: the device filter was accepted
                self.reader = threading.Thread(target=self._read, daemon=True)
                self.reader.start()
                break
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _to_torch(a: np.ndarray):
    """Host array -> CPU tensor over the same memory (uint16 = bf16 bits)."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


class Problem:
    """Device buffers, one raw C-ABI launch closure and the same operation
    through the public tensor API (for the end-to-end measurement) for a named
    workload."""

    def __init__(self, workload: str, fmt: str, dev, seed: int = 0, sf_flags: int = 0,
                 like: "Problem | None" = None, row_begin: int = 0):
        """`like`: another Problem of the same workload whose inputs are copied
        to new device buffers (a second buffer set of the same launch, for the
        sustained timing); `row_begin`: the first row of this rank's shard of a
        multi-GPU batch (rows [row_begin, row_begin + T) of one longer draw)."""
        import torch
        import fp8_activation_quantization_gb300 as tkq
        from fp8_activation_quantization_gb300 import synth
        self.workload = workload
        self.kern = kern = KERNEL_OF[workload]
        self.fmt = fmt
        self.sf_flags = sf_flags
        if like is not None:
            self.host = like.host
        else:
            self.host = synth.workload(SYNTH_OF.get(workload, workload), seed=seed,
                                       row_begin=row_begin)
        lead = self.host["x"] if "x" in self.host else self.host["codes"]
        self.T, self.C = T, C = lead.shape
        self.weighted = "w" in self.host
        self.bytes = algorithmic_bytes(workload, T, C, self.weighted)
        self.dev = dev
        if like is not None:
            self.inp = {k: v.clone() for k, v in like.inp.items()}
        else:
            self.inp = {k: _to_torch(v).to(dev) for k, v in self.host.items()}
        fcode = 0 if fmt == "e4m3" else 1
        fp8 = _fp8(fmt)
        P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        x, w, dy = self.inp.get("x"), self.inp.get("w"), self.inp.get("dy")
        u8, f32 = torch.uint8, torch.float32
        E = lambda shape, dt=u8: torch.empty(shape, dtype=dt, device=dev)
        opt = dict(round_sf=bool(sf_flags & 1), use_packed_ue8m0=bool(sf_flags & 2),
                   use_tma_aligned_col_major_sf=bool(sf_flags & 4))
        sf_done = False   # a branch that handles sf_flags itself
        if kern == "per_token_cast":
            self.outputs = [E((T, C)), E((T, C // 128), f32)]
            fn, args = tkq.tkq_per_token_cast, [P(x), P(self.outputs[0]), None, T, C, 128, fcode]
            sf_pos = 2
            self.api = lambda i, od: tkq.per_token_cast(i["x"], fmt, out=od[0].view(fp8),
                                                        out_sf=od[1], **opt)
        elif kern == "swiglu_cast":
            H = C // 2
            self.outputs = [E((T, H)), E((T, H // 128), f32)]
            fn, args = tkq.tkq_swiglu_cast, [P(x), P(w), P(self.outputs[0]), None, T, H, 128,
                                             fcode]
            sf_pos = 3
            self.api = lambda i, od: tkq.swiglu_forward_and_per_token_cast(
                i["x"], fmt, topk_weights=i.get("w"), out=od[0].view(fp8), out_sf=od[1], **opt)
        elif kern == "per_token_cast_f32":
            self.outputs = [E((T, C)), E((T, C // 128), f32)]
            fn, args = tkq.tkq_per_token_cast_f32, [P(x), P(self.outputs[0]), None, T, C, 128,
                                                    fcode, sf_flags]
            sf_pos = 2
            self.api = lambda i, od: tkq.per_token_cast(i["x"], fmt, out=od[0].view(fp8),
                                                        out_sf=od[1], **opt)
        elif kern == "swiglu_cast_clamp":
            H = C // 2
            self.count = E((1,), torch.int64).zero_()
            self.outputs = [E((T, H)), E((T, H // 128), f32)]
            fn, args = tkq.tkq_swiglu_cast_clamp, [P(x), P(w), P(self.outputs[0]), None, T, H,
                                                   128, fcode, sf_flags, CLAMP_VALUE,
                                                   P(self.count)]
            sf_pos = 3
            self.api = lambda i, od: tkq.swiglu_forward_and_per_token_cast(
                i["x"], fmt, topk_weights=i.get("w"), out=od[0].view(fp8), out_sf=od[1],
                use_clamp=True, swiglu_clamp_value=CLAMP_VALUE, clamp_count=self.count, **opt)
        elif kern == "swiglu_backward_cast":
            H = C // 2
            self.outputs = [E((T, 2 * H)), E((T, 2 * H // 128), f32)]
            fn, args = tkq.tkq_swiglu_backward_cast, [P(x), P(dy), P(w), P(self.outputs[0]),
                                                      None, T, H, 128, fcode]
            sf_pos = 4
            self.api = lambda i, od: tkq.swiglu_backward_and_per_token_cast(
                i["x"], i["dy"], fmt, topk_weights=i.get("w"), out=od[0].view(fp8),
                out_sf=od[1], **opt)
        elif kern == "swiglu_cast_t":
            H = C // 2
            if sf_flags:
                # both scale outputs in the layout the flags select
                self.outputs = [E((T, H)), E((tkq.tkq_sf_bytes(T, H // 128, sf_flags),)),
                                E((H, T)), E((tkq.tkq_sf_bytes(H, T // 128, sf_flags),))]
            else:
                self.outputs = [E((T, H)), E((T, H // 128), f32), E((H, T)),
                                E((H, T // 128), f32)]
            o = self.outputs
            args = [P(x), P(w), P(o[0]), P(o[1]), P(o[2]), P(o[3]), T, H, 128, fcode]
            if sf_flags:
                fn = tkq.tkq_swiglu_cast_t_ex
                args.append(sf_flags)
            else:
                fn = tkq.tkq_swiglu_cast_t
            sf_pos = None
            sf_done = True
            self.api = lambda i, od: tkq.swiglu_forward_and_per_token_cast(
                i["x"], fmt, topk_weights=i.get("w"), with_transpose=True,
                out=od[0].view(fp8), out_sf=od[1], out_t=od[2].view(fp8), out_sf_t=od[3], **opt)
        elif kern == "swiglu_cast_t_clamp":
            H = C // 2
            self.count = E((1,), torch.int64).zero_()
            self.outputs = [E((T, H)), E((T, H // 128), f32), E((H, T)), E((H, T // 128), f32)]
            o = self.outputs
            fn, args = tkq.tkq_swiglu_cast_t_clamp, [P(x), P(w), P(o[0]), P(o[1]), P(o[2]),
                                                     P(o[3]), T, H, 128, fcode, 0, CLAMP_VALUE,
                                                     P(self.count)]
            sf_pos = None
            self.api = lambda i, od: tkq.swiglu_forward_and_per_token_cast(
                i["x"], fmt, topk_weights=i.get("w"), with_transpose=True,
                out=od[0].view(fp8), out_sf=od[1], out_t=od[2].view(fp8), out_sf_t=od[3],
                use_clamp=True, swiglu_clamp_value=CLAMP_VALUE, clamp_count=self.count)
        elif kern in ("per_channel_cast", "per_channel_cast_t"):
            tr = kern.endswith("_t")
            self.outputs = [E((C, T) if tr else (T, C)),
                            E((C, T // 128) if tr else (T // 128, C), f32)]
            fn, args = tkq.tkq_per_channel_cast, [P(x), P(self.outputs[0]), P(self.outputs[1]),
                                                  T, C, 128, fcode, int(tr)]
            sf_pos = None
            self.api = lambda i, od: tkq.per_channel_cast(i["x"], fmt, transpose=tr,
                                                          out=od[0].view(fp8), out_sf=od[1])
        elif kern == "per_block_cast":
            self.outputs = [E((T, C)), E((-(-T // 128), C // 128), f32)]
            fn, args = tkq.tkq_per_block_cast, [P(x), P(self.outputs[0]), P(self.outputs[1]),
                                                T, C, 128, fcode]
            sf_pos = None
            self.api = lambda i, od: tkq.per_block_cast(i["x"], fmt, out=od[0].view(fp8),
                                                        out_sf=od[1])
        elif kern == "cast_back":
            self.outputs = [E((T, C), torch.bfloat16)]
            fn, args = tkq.tkq_cast_back, [P(self.inp["codes"]), P(self.inp["sf"]),
                                           P(self.outputs[0]), T, C, 1, 128, fcode, tkq.OUT_BF16]
            sf_pos = None
            self.api = lambda i, od: (tkq.cast_back(i["codes"], i["sf"], fmt=fmt,
                                                    group_size=(1, 128),
                                                    out_dtype=torch.bfloat16, out=od[0]),)
        else:
            raise KeyError(kern)
        if sf_pos is not None and kern in ("swiglu_cast_clamp", "per_token_cast_f32"):
            if sf_flags:
                G = self.outputs[1].numel() // T
                self.outputs[1] = E((tkq.tkq_sf_bytes(T, G, sf_flags),))
            args[sf_pos] = P(self.outputs[1])
        elif sf_pos is not None:
            if sf_flags:
                # the same kernel with a scale-factor layout: the _ex call
                G = self.outputs[1].numel() // T
                self.outputs[1] = E((tkq.tkq_sf_bytes(T, G, sf_flags),))
                args.append(sf_flags)
                fn = {"per_token_cast": tkq.tkq_per_token_cast_ex,
                      "swiglu_cast": tkq.tkq_swiglu_cast_ex,
                      "swiglu_backward_cast": tkq.tkq_swiglu_backward_cast_ex}[kern]
            args[sf_pos] = P(self.outputs[1])
        elif sf_flags and not sf_done:
            raise ValueError("scale-layout options apply to the row and transposed casts only")
        self._fn, self._args = fn, tuple(args)

    def launch(self, stream):
        st = self._fn(*self._args, ctypes.c_void_p(stream.cuda_stream))
        if st:
            raise RuntimeError(f"{self.kern} failed with status {st}")


def time_flushed(prob: Problem, reps: int, stream, flush):
    """Median per-launch time with L2 flushed before each launch.  The flush
    READS a buffer four times the size of L2, which leaves L2 full of clean
    lines (a write-based flush would leave dirty lines whose write-back lands
    inside the timed launch)."""
    import torch
    ts = []
    for i in range(reps + 3):
        flush.max()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        prob.launch(stream)
        e.record(stream)
        e.synchronize()
        if i >= 3:
            ts.append(s.elapsed_time(e) / 1000.0)
    return float(np.median(ts))


SMALL_BYTES = 512e6  # below this the working set could stay in L2 between steps
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (the ~8 TB/s the 80 % bar refers to)


def l2_bytes(dev) -> int:
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size) or 129 << 20
    except Exception:
        return 129 << 20


def rotation_sets(prob: Problem, l2: int) -> int:
    """Buffer sets the sustained timing rotates over: enough that their inputs
    and outputs together span at least four times L2, and at least two."""
    return max(2, -(-4 * l2 // max(prob.bytes, 1)))


def time_sustained(probs, stream, min_launches: int = 200):
    """Per-launch time (seconds) of launches issued back to back over a rotation
    of buffer sets (the Problems in `probs`, one per set).  With the sets
    spanning several times L2, every launch reads inputs that are not in L2,
    and the write-back of each launch's output is paid inside the launches that
    follow it, as in a stream of casts; only the last launch's dirty lines fall
    outside the timed region, one launch's worth over all of them.  The
    launches (a multiple of the rotation, at least `min_launches`) are captured
    in one CUDA graph and replayed, so that host launch cost cannot pace short
    kernels; one warm-up pass over the rotation and one warm-up replay come
    first.  Returns (seconds per launch, launches timed)."""
    import torch
    k = len(probs)
    n = max(1, -(-min_launches // k)) * k
    for p in probs:
        p.launch(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(n):
            probs[i % k].launch(stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    e.record(stream)
    e.synchronize()
    dt = s.elapsed_time(e) / 1000.0 / n
    del g
    return dt, n


class CopyProblem:
    """A device-to-device copy moving the same bytes as one launch of a
    workload (half read, half written): what the memory system gives a launch
    of that size, timed the same way as the kernel."""

    def __init__(self, nbytes: int, dev):
        import torch
        n = max(16, nbytes // 2)
        self.src = torch.empty(n, dtype=torch.uint8, device=dev)
        self.dst = torch.empty_like(self.src)
        self.bytes = 2 * n

    def launch(self, stream):
        import torch
        with torch.cuda.stream(stream):
            self.dst.copy_(self.src)


def copy_rotation(nbytes: int, dev, l2: int):
    first = CopyProblem(nbytes, dev)
    return [first] + [CopyProblem(nbytes, dev)
                      for _ in range(max(2, -(-4 * l2 // first.bytes)) - 1)]


def rotation(prob: Problem, l2: int):
    """The buffer sets of a sustained timing: `prob` and copies of it."""
    sets = [prob]
    for _ in range(rotation_sets(prob, l2) - 1):
        sets.append(Problem(prob.workload, prob.fmt, prob.dev, sf_flags=prob.sf_flags, like=prob))
    return sets


def rank_shard(workload: str, ws: int, rank: int, rows: int | None = None) -> tuple[int, int, int]:
    """Weak scaling over `ws` ranks: the global batch is `ws` times the
    workload's rows (or `rows` per rank), split by shard_rows into contiguous
    ranges (multiples of 128 rows where the row count allows, so the transposed
    cast's 128-token groups never straddle two ranks).  Returns (first row, end
    row, global rows) of this rank's shard."""
    from fp8_activation_quantization_gb300 import synth
    from fp8_activation_quantization_gb300.sharding import shard_rows
    T = synth.WORKLOADS[SYNTH_OF.get(workload, workload)][0] if rows is None else int(rows)
    align = 128 if T % 128 == 0 else 1
    a, b = shard_rows(T * ws, ws, rank, align)
    return a, b, T * ws


def e2e_steps(prob: Problem, steps: int, stream):
    """Metric through the public tensor API with host buffers.  Every step
    copies its inputs from pinned host memory to the device, runs the op and
    copies every output back to pinned host memory.  Copy-in, compute and
    copy-out run on three streams over two device buffer sets, so step i+1's
    copy-in overlaps step i's compute and copy-out (as a user streaming batches
    would run it); the timed region spans the first copy-in to the last
    copy-out."""
    import torch
    dev = prob.dev
    pin = {k: _to_torch(v).pin_memory() for k, v in prob.host.items()}
    outs_pin = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in prob.outputs]
                for _ in range(2)]
    inp_dev = [{k: torch.empty_like(v, device=dev) for k, v in pin.items()} for _ in range(2)]
    outs_dev = [[torch.empty_like(o) for o in prob.outputs] for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(o.numel() * o.element_size() for o in prob.outputs)
    s_in, s_out, s_cmp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), stream
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(cmp_done[b])      # step i-2 finished reading the inputs of set b
        with torch.cuda.stream(s_in):
            for k, v in pin.items():
                inp_dev[b][k].copy_(v, non_blocking=True)
            in_done[b].record(s_in)
        s_cmp.wait_event(in_done[b])
        if i >= 2:
            s_cmp.wait_event(out_done[b])     # step i-2's outputs have left the device
        with torch.cuda.stream(s_cmp):
            res = prob.api(inp_dev[b], outs_dev[b])
            cmp_done[b].record(s_cmp)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            for hp, dv in zip(outs_pin[b], res):
                hp.copy_(dv.view(hp.dtype) if dv.dtype != hp.dtype else dv, non_blocking=True)
            out_done[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        step(i)
    end.record(s_out)
    torch.cuda.synchronize()
    dt = start.elapsed_time(end) / 1000.0
    return dt, h2d, d2h


def _fp8(fmt):
    import torch
    return torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2


def run_oracle(kern: str, d: dict, rows: int, fmt: str, threads: int = 1):
    """The oracle for one kernel on the first `rows` rows of a workload dict."""
    import oracle
    if kern == "cast_back":
        import torch
        y = oracle.cast_back(d["codes"][:rows], d["sf"][:rows], 1, 128, fmt, threads=threads)
        return torch.from_numpy(y).to(torch.bfloat16)
    x = d["x"][:rows]
    w = None if d.get("w") is None else d["w"][:rows]
    if kern in ("per_channel_cast", "per_channel_cast_t"):
        return oracle.per_channel_cast(x, fmt, transpose=kern.endswith("_t"), threads=threads)
    if kern == "per_block_cast":
        return oracle.per_block_cast(x, fmt, threads=threads)
    if kern == "per_token_cast":
        return oracle.per_token_cast(x, fmt, threads=threads)
    if kern == "per_token_cast_f32":
        return oracle.cast_rows_f32_ex(x, fmt, threads=threads)
    if kern == "swiglu_cast":
        return oracle.swiglu_cast(x, w, fmt, threads=threads)
    if kern == "swiglu_cast_clamp":
        return oracle.swiglu_cast(x, w, fmt, threads=threads, clamp=CLAMP_VALUE)
    if kern == "swiglu_backward_cast":
        return oracle.swiglu_backward_cast(x, d["dy"][:rows], w, fmt, threads=threads)
    if kern == "swiglu_cast_t_clamp":
        return oracle.swiglu_cast_t(x, w, fmt, threads=threads, clamp=CLAMP_VALUE)
    return oracle.swiglu_cast_t(x, w, fmt, threads=threads)


def _lead(d: dict) -> np.ndarray:
    """The array whose rows are the workload's tokens."""
    return d["x"] if "x" in d else d["codes"]


CPU_BASELINE_SECONDS = 10.0   # at least this much oracle time per cpu_baseline
CPU_BASELINE_BLOCK = 8192     # rows per oracle call (a multiple of 128)


def cpu_baseline_single_thread(workload: str, fmt: str, host: dict | None = None,
                               min_seconds: float = CPU_BASELINE_SECONDS):
    """The oracle, as it stands, on one host core: consecutive blocks of
    CPU_BASELINE_BLOCK rows of the workload, from its first row, until at least
    `min_seconds` of oracle time are spent or the workload is exhausted."""
    from fp8_activation_quantization_gb300 import synth
    d = host if host is not None else synth.workload(SYNTH_OF.get(workload, workload))
    T, C = _lead(d).shape
    kern = KERNEL_OF[workload]
    done, spent = 0, 0.0
    while done < T and spent < min_seconds:
        end = min(T, done + CPU_BASELINE_BLOCK)
        part = {k: np.ascontiguousarray(v[done:end]) for k, v in d.items()}
        t0 = time.perf_counter()
        run_oracle(kern, part, end - done, fmt)
        spent += time.perf_counter() - t0
        done = end
    b = algorithmic_bytes(workload, done, C, "w" in d)
    return {"value": round(b / spent / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {done} rows of the {workload} workload ({b / 1e6:.0f} MB of "
                      f"algorithmic bytes) in blocks of {CPU_BASELINE_BLOCK} rows, "
                      f"single-threaded C oracle, {spent:.1f} s",
            "rows_per_s": round(done / spent, 1)}


def max_over_ranks(dt: float, ws: int, dev=None) -> float:
    """The slowest rank's time (every rank gets it)."""
    if ws <= 1:
        return dt
    import torch
    import torch.distributed as dist
    t = torch.tensor([dt], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {ws}")
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = lambda: dist.barrier()
    else:
        barrier = lambda: None
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if ws > 1:
        barrier()
    import fp8_activation_quantization_gb300 as tkq
    tkq.load_library()
    stream = torch.cuda.Stream(dev)
    peak, peak_src = measured_peaks()

    # this rank's shard of a batch of ws workloads' worth of rows (weak scaling)
    row0, row1, rows_global = rank_shard(args.workload, ws, rank)
    prob = Problem(args.workload, args.fmt, dev, row_begin=row0, sf_flags=args.sf_flags)
    assert prob.T == row1 - row0
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    tkq.tkq_read_device_status(clear=True)
    small = prob.bytes < SMALL_BYTES
    l2 = l2_bytes(dev)
    sets = rotation(prob, l2) if small else [prob]
    with torch.cuda.stream(stream):
        with ClockSampler(uuid) as clk:
            dt = time_rotation(sets, args.steps, args.warmup, stream, barrier)
        # the same launches issued one by one from the host, for comparison
        dt_stream = time_rotation(sets, min(args.steps, 200), 0, stream, barrier, graph=False)
        dt_stream *= args.steps / min(args.steps, 200)
    if tkq.tkq_read_device_status():
        raise RuntimeError("a bounded wait inside a kernel gave up: timing is invalid")
    dt = max_over_ranks(dt, ws, dev)
    dt_stream = max_over_ranks(dt_stream, ws, dev)
    total_bytes = prob.bytes * args.steps * ws
    gbs = total_bytes / dt / 1e9
    per_launch = dt / args.steps
    achieved = prob.bytes / per_launch / 1e9
    rows_per_s = prob.T * args.steps * ws / dt

    if rank != 0:
        if ws > 1:
            barrier()
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    res = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded, generated on the host; see config.workload)",
        "config": workload_config(args.workload, args.fmt, ws),
        "buffer_sets": len(sets),
        "pct_of_peak": round(100.0 * gbs / ws / peak, 2),
        "pct_of_nominal_peak": round(100.0 * gbs / ws / NOMINAL_HBM_GBS, 2),
        "rows_per_s": round(rows_per_s, 1),
        "gpu_launches": args.steps,
        "launch": "the K timed launches captured in one CUDA graph, timed as one replay",
        "ms_per_step_stream_launches": round(dt_stream / args.steps * 1e3, 5),
        "clocks": clk.summary(),
        "roofline": {
            "bound": "hbm", "kernel": prob.kern,
            "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(prob.kern, args.workload),
            "algorithmic_bytes_per_launch": prob.bytes,
            "peak_source": peak_src,
            "nominal_peak": NOMINAL_HBM_GBS,
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
        },
    }
    if ws > 1:
        res["shards"] = {"rows_per_rank": prob.T, "rows_global": rows_global,
                         "rank0_rows": [row0, row1]}
    del sets
    if not args.no_extras and ws == 1:
        e_steps = max(3, min(args.steps, 20))
        edt, h2d, d2h = e2e_steps(prob, e_steps, stream)
        res["e2e"] = {"value": round(prob.bytes * e_steps / edt / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": round(edt / e_steps * 1e3, 3)}
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if small else None
        with torch.cuda.stream(stream):
            tc = d2d_copy_reference(prob, stream, flush)
        del flush
        res["d2d_copy"] = {"us": round(tc * 1e6, 2), "GB/s": round(prob.bytes / tc / 1e9, 1),
                           "bytes": prob.bytes - prob.bytes % 2,
                           "kernel_time_over_copy_time": round(per_launch / tc, 3),
                           "note": "cudaMemcpyAsync device-to-device of half the algorithmic "
                                   "bytes (read + write = the same traffic), timed like the kernel"}
        res["cpu_baseline"] = cpu_baseline_single_thread(args.workload, args.fmt, prob.host)
        del prob
        torch.cuda.empty_cache()
        res["per_workload"] = other_workloads(dev, stream, peak, args)
        res["bar_80pct"] = bar_table(res["per_workload"], peak)
    print(json.dumps(res), flush=True)
    if ws > 1:
        barrier()
        import torch.distributed as dist
        dist.destroy_process_group()


def time_rotation(sets, steps: int, warmup: int, stream, barrier, graph: bool = True) -> float:
    """K timed launches (seconds, CUDA events around the whole run) back to
    back, launch i on buffer set i mod len(sets); W untimed launches first.
    With one set this is plain back-to-back timing (inputs larger than L2).
    graph: the K launches are captured in one CUDA graph and the timed region
    is its replay (the warm-up launches run before the capture, and one
    untimed replay after it); otherwise each launch is issued from the host
    inside the timed region."""
    import torch
    k = len(sets)
    for i in range(max(warmup, k)):
        sets[i % k].launch(stream)
    torch.cuda.synchronize()
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(steps):
                sets[i % k].launch(stream)
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    if graph:
        with torch.cuda.stream(stream):
            g.replay()
    else:
        for i in range(steps):
            sets[i % k].launch(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / 1000.0


# the 80 % bar of the plain and fused casts at T >= 8192, judged on the
# sustained (write-back inclusive) rate
BAR_WORKLOADS = ["plain_outlier/e4m3", "plain_outlier/e5m2", "swiglu/e4m3",
                 "swiglu_moe/e4m3", "swiglu_t/e4m3"]


def bar_table(per_workload: dict, peak: float) -> dict:
    out = {}
    for key in BAR_WORKLOADS:
        e = per_workload.get(key)
        if not e:
            continue
        gbs = e["sustained"]["GB/s"]
        out[key] = {"GB/s_sustained": gbs, "frac_of_measured": round(gbs / peak, 4),
                    "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                    "pass_measured": gbs >= 0.8 * peak,
                    "pass_nominal": gbs >= 0.8 * NOMINAL_HBM_GBS}
    return out


def d2d_copy_reference(prob: Problem, stream, flush):
    """A device-to-device cudaMemcpyAsync (torch copy_) moving the same bytes
    as one launch (half read, half written), timed like the kernel: median of
    L2-flushed copies for small problems, back-to-back copies otherwise."""
    import torch
    n = prob.bytes // 2
    src = torch.empty(n, dtype=torch.uint8, device=prob.dev)
    dst = torch.empty_like(src)
    ts = []
    for i in range(13):
        if flush is not None:
            flush.max()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        dst.copy_(src)
        e.record(stream)
        e.synchronize()
        if i >= 3:
            ts.append(s.elapsed_time(e) / 1000.0)
    t = float(np.median(ts))
    return t


def other_workloads(dev, stream, peak, args):
    """Each kernel on every workload shape, timed two ways: `us`, the median of
    single launches each preceded by an L2 flush (a cold start; the launch's
    own write-back is partly left to the next flush), and `sustained`, launches
    back to back over a rotation of buffer sets spanning four times L2 (every
    launch's write-back paid inside the timed region, as in a stream of casts;
    see time_sustained)."""
    import torch
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    l2 = l2_bytes(dev)
    out = {}
    for name, fmt, flags in [("plain_small", "e4m3", 0), ("plain_outlier", "e4m3", 0),
                             ("plain_outlier", "e5m2", 0), ("plain_outlier", "e4m3", 6),
                             ("plain_outlier", "e4m3", 8),
                             ("swiglu", "e4m3", 0), ("swiglu", "e4m3", 6),
                             ("swiglu_moe", "e4m3", 0),
                             ("swiglu_moe", "e4m3", 6), ("swiglu_t", "e4m3", 0),
                             ("swiglu_t", "e4m3", 6),
                             ("swiglu_bwd", "e4m3", 0), ("per_channel", "e4m3", 0),
                             ("per_channel_t", "e4m3", 0), ("per_block", "e4m3", 0),
                             ("cast_back", "e4m3", 0), ("swiglu_clamp", "e4m3", 0),
                             ("swiglu_t_clamp", "e4m3", 0), ("plain_f32", "e4m3", 0)]:
        prob = Problem(name, fmt, dev, sf_flags=flags)
        with torch.cuda.stream(stream):
            t = time_flushed(prob, 20, stream, flush)
            sets = rotation(prob, l2)
            ts, n = time_sustained(sets, stream)
            k = len(sets)
            del sets
            copies = copy_rotation(prob.bytes, dev, l2)
            tc, _ = time_sustained(copies, stream)
            del copies
        gbs = prob.bytes / t / 1e9
        gbs_s = prob.bytes / ts / 1e9
        key = f"{name}/{fmt}" + {0: "", 6: "/ue8m0-col-major-sf", 8: "/sf-inv"}[flags]
        out[key] = {"kernel": prob.kern, "us": round(t * 1e6, 2),
                    "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                    "rows_per_s": round(prob.T / t, 1), "bytes": prob.bytes,
                    "sustained": {"us": round(ts * 1e6, 2), "GB/s": round(gbs_s, 1),
                                  "frac": round(gbs_s / peak, 4),
                                  "frac_of_nominal": round(gbs_s / NOMINAL_HBM_GBS, 4),
                                  "buffer_sets": k, "launches": n,
                                  "copy_us": round(tc * 1e6, 2),
                                  "kernel_time_over_copy_time": round(ts / tc, 3)}}
        del prob
        torch.cuda.empty_cache()
    return out


def workload_config(workload: str, fmt: str, ws: int) -> dict:
    """The `config` object of the JSON line: the same for both arms."""
    from fp8_activation_quantization_gb300 import synth
    syn = SYNTH_OF.get(workload, workload)
    T, C, _ = synth.WORKLOADS[syn]
    weighted = "w" in synth.workload(syn, rows=1)
    nbytes = algorithmic_bytes(workload, T, C, weighted)
    if nbytes < SMALL_BYTES:
        l2 = ("launches back to back over a rotation of buffer sets (inputs and outputs; "
              "buffer_sets of them) spanning at least 4x L2: every launch reads inputs "
              "not in L2 and pays the write-back of earlier launches")
    else:
        l2 = "inputs larger than L2 (no flush between steps)"
    return {
        "workload": _workload_desc(workload),
        "T": T, "cols": C, "fmt": fmt, "group": 128,
        "weighted": weighted,
        "algorithmic_bytes_per_step": nbytes,
        "l2": l2,
        "parallelism": (f"dp{ws}: each rank quantizes its own {T}-row shard of a "
                        f"{T * ws}-row batch (rows independent, no collective)"
                        if ws > 1 else "single GPU (rows independent, no collective)"),
    }


def _workload_desc(name):
    from fp8_activation_quantization_gb300 import synth
    d = synth.WORKLOADS[SYNTH_OF.get(name, name)][2]
    if name == "per_channel_t":
        return d.replace("per_channel_cast (+transpose)", "per_channel_cast + transpose")
    if name.endswith("_clamp"):
        return d.replace("swiglu +", f"swiglu with clamp c = {CLAMP_VALUE:g} (count kept) +", 1)
    return d


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from fp8_activation_quantization_gb300 import synth
    oracle.build()
    cores = max(1, os.cpu_count() or 1)
    syn = SYNTH_OF.get(args.workload, args.workload)
    T_full, C, _ = synth.WORKLOADS[syn]
    kern = KERNEL_OF[args.workload]
    # calibrate: one 128-row block per core
    rows = 128 * cores
    d = synth.workload(syn, rows=min(T_full, 8192))
    x_all, w_all = _lead(d), d.get("w")

    def step(r):
        run_oracle(kern, d, r, args.fmt, threads=cores)

    t0 = time.perf_counter()
    step(min(rows, x_all.shape[0]))
    t_cal = time.perf_counter() - t0
    per_row = t_cal / min(rows, x_all.shape[0])
    budget = args.ref_seconds  # seconds for warmup + steps
    r = int(budget / max(args.steps + args.warmup, 1) / per_row)
    r = max(128, min(x_all.shape[0], (r // 128) * 128))
    for _ in range(args.warmup):
        step(r)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(r)
    dt = time.perf_counter() - t0
    b = algorithmic_bytes(args.workload, r, C, w_all is not None)
    gbs = b * args.steps / dt / 1e9
    res = {
        "impl": "reference",
        "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, generated on the host; see config.workload)",
        "config": workload_config(args.workload, args.fmt, ws),
        "rows_per_s": round(r * args.steps / dt, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {r} rows of the workload per step, row blocks split "
                                   f"over {cores} threads"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def launch_ranks(args) -> int:
    """--gpus N > 1 outside torchrun: start N ranks on this node, one per GPU,
    through torch.distributed.run, or fail when the node has fewer GPUs."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(KERNEL_OF))
    ap.add_argument("--fmt", default="e4m3", choices=["e4m3", "e5m2"])
    ap.add_argument("--no-extras", action="store_true",
                    help="skip e2e, CPU baseline and the per-workload table")
    ap.add_argument("--sf-flags", type=int, default=0,
                    help="scale-layout flags (TKQ_SF_*) of the timed cast")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: oracle time to aim for over warmup + steps")
    args = ap.parse_args()
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be >= 1")
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "ours":
        import torch
        have = torch.cuda.device_count()
        if have < args.gpus:
            print(f"bench.py: --gpus {args.gpus} needs {args.gpus} GPUs, {have} visible",
                  file=sys.stderr)
            sys.exit(2)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
