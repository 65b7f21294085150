#!/usr/bin/env python
"""Throughput of the GB300 sum-reduction library on its workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

A step is one pass of every reduction entry point over its workload's input:
  fp32 sum and sum of squares of n = 2^24 + 13 normal(0,1) values (seed 1),
  int32 -> int64 sum of n = 2^28 uniform integers in [-2^20, 2^20] (seed 2),
  fp32 row sums of 8192 x 32768 and of 2^20 x 256 uniform[-1,1) (seed 3),
  bf16 -> fp32 sum and sum of squares of n = 2^30 + 7 normal(0,1) (seed 4).
The metric is GB/s of input read by the reductions (algorithmic bytes / device
time).  Every launch is timed with CUDA events on the stream it runs on, after
an untimed L2 flush (a 512 MiB write, then a 512 MiB read so that the timed
kernel finds no dirty line to write back), so each launch reads its input from
HBM.  ``e2e`` repeats the step from pinned host memory: the
host-to-device copies of the inputs and the device-to-host copies of the
results are inside its timed region.  ``cpu_baseline`` times the CPU oracle
(one core) on a bounded sample of the same step.

After the timed region every step's results, and the host copies of the last
end-to-end step, are compared with the CPU oracle over the whole input
(bit-exact for the int32 sum, within the float tolerances otherwise, per row
for row sums), and the steps must agree bit for bit; the line's ``parity``
object reports it and the exit status is 1 on any mismatch.

``--impl reference`` times the CPU oracle alone, as the comparison arm, on a
bounded sample of each step.

Under torchrun each rank reduces its own copy of the workload (weak scaling,
no collective on the data path); the time is the maximum over ranks.  The
line's ``sharded`` object then also times the bf16 and int32 sums split over
the ranks (strong scaling: a chunk per rank, an NCCL all-gather of the
partials, the rank-order combine).  On one GPU, ``extras`` times that split
over 8 chunks emulated on the one device.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from reduction_rdx_sum_gb300 import inputs  # noqa: E402

METRIC = "reduction GB/s read (and % of GB300 HBM peak) per config, 1 GPU"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# (profiles/ has the summaries), with the source files that define the kernel
# and their hash at capture time: a figure is reported only while those files
# are unchanged.  The captures ran on n = 2^28 and are scaled to the full launch
# by the element count (traffic grows in proportion).
_RED = ("device.cuh", "reduce.cu")
_ROW = ("device.cuh", "rowsum.cu")
_RED_HASH = "64a04e1696a0e1b1"
_ROW_HASH = "7712c0542427d0a1"
NCU_TRAFFIC = {
    # workload: bytes per full launch, scaled from the capture named in the profile
    "c5_sum_bf16": {"bytes_per_launch": 2160423950, "sources": _RED, "source_hash": _RED_HASH,
                    "profile": "profiles/reduce_kernel_SumBF16_bf16_n268435456.md"},
    "c5_sumsq_bf16": {"bytes_per_launch": 2158738446, "sources": _RED, "source_hash": _RED_HASH,
                      "profile": "profiles/kernels_dram_traffic_small_cases.md"},
    "c3_sum_i32": {"bytes_per_launch": 1078776832, "sources": _RED, "source_hash": _RED_HASH,
                   "profile": "profiles/kernels_dram_traffic_small_cases.md"},
    "c2_sum_f32": {"bytes_per_launch": 67197440, "sources": _RED, "source_hash": _RED_HASH,
                   "profile": "profiles/kernels_dram_traffic_small_cases.md"},
    "c4_rowsum_8192x32768": {"bytes_per_launch": 1079667712, "sources": _ROW, "source_hash": _ROW_HASH,
                             "profile": "profiles/kernels_dram_traffic_small_cases.md"},
    "c4_rowsum_1048576x256": {"bytes_per_launch": 1086131200, "sources": _ROW, "source_hash": _ROW_HASH,
                              "profile": "profiles/kernels_dram_traffic_small_cases.md"},
}


def code_tokens(text: str) -> str:
    """C++ source with comments removed and whitespace collapsed: what the
    compiler sees, so that editing a comment does not read as a kernel change."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(files=None) -> str:
    """Hash of the kernel sources' code (all of csrc/, or the named files),
    comments and layout excluded."""
    csrc = os.path.join(ROOT, "reduction_rdx_sum_gb300", "csrc")
    names = sorted(files) if files else sorted(os.listdir(csrc))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    t = NCU_TRAFFIC.get(workload)
    if t and kernel_source_hash(t["sources"]) == t["source_hash"]:
        return t["bytes_per_launch"]
    return None


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    """Largest value over all ranks (timing is reported for the slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------

def suite_arrays():
    """Host inputs of the step; workloads that share a recipe share an array."""
    arrays, keyed = {}, {}
    for w in inputs.SUITE:
        key = (w.dist, w.seed, w.numel)
        if key not in keyed:
            keyed[key] = inputs.make(w).reshape(-1)
        arrays[w.name] = keyed[key]
    return arrays, keyed


def step_bytes():
    return sum(w.bytes_read for w in inputs.SUITE)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None):
        self.path = path
        self.proc = None
        self.gpu_index = gpu_index

    def __enter__(self):
        try:
            self.out = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu_index)], stdout=self.out, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                text = self.proc.communicate(timeout=5)[0] if not self.path else None
            except subprocess.TimeoutExpired:
                self.proc.kill()
                text = None
            if self.path:
                self.out.close()
                with open(self.path) as f:
                    text = f.read()
            self.text = text or ""
        else:
            self.text = ""

    def summary(self):
        rows = [r.split(",") for r in self.text.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        power = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (the reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_pass(arrays, frac: float):
    """Run the oracle over the first `frac` of every workload of the step;
    returns (bytes processed, seconds)."""
    import oracle

    total, t0 = 0, time.perf_counter()
    for w in inputs.SUITE:
        a = arrays[w.name]
        if w.op == "rowsum_f32":
            rows, cols = w.shape
            r = max(1, int(rows * frac))
            oracle.rowsum_f32(a[: r * cols].reshape(r, cols))
            total += r * cols * 4
            continue
        k = max(1, int(a.size * frac))
        getattr(oracle, w.op)(a[:k])
        total += k * w.itemsize
    return total, time.perf_counter() - t0


def calibrate_oracle(arrays, budget_s: float):
    """Fraction of the step the oracle finishes in about budget_s seconds."""
    b, s = oracle_pass(arrays, 1.0 / 256)
    rate = b / max(s, 1e-9)
    return min(1.0, budget_s * rate / step_bytes())


def cpu_threads_rate(arrays):
    """The oracle's loops on every host core (oracle/threads.c): one
    contiguous chunk per thread, float64 Kahan or int64 per chunk, chunk
    results added in fixed order; row sums split by rows.  The whole step,
    reported beside the single-thread oracle rate as a second CPU baseline."""
    import oracle

    threads = oracle.default_threads()
    t0 = time.perf_counter()
    for w in inputs.SUITE:
        a = arrays[w.name]
        if w.op == "rowsum_f32":
            oracle.threaded_rowsum_f32(a.reshape(w.shape), threads)
        else:
            oracle.threaded(w.op, a, threads)
    secs = time.perf_counter() - t0
    return {"value": round(step_bytes() / secs / 1e9, 2), "unit": UNIT, "cores": threads,
            "host_cores": os.cpu_count(), "kind": "oracle, threaded (one contiguous chunk per core)",
            "sample": "the whole step", "seconds": round(secs, 2)}


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle, as it stands, on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import oracle

    oracle.build()
    arrays, _ = suite_arrays()
    # about 150 s of oracle work for the whole run, at most 10 s per step
    per_step_budget = max(0.5, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    per_step_budget = float(os.environ.get("RDX_BENCH_REFERENCE_BUDGET_S", per_step_budget))
    frac = calibrate_oracle(arrays, per_step_budget)
    for _ in range(args.warmup):
        oracle_pass(arrays, frac)
    done, secs = 0, 0.0
    for _ in range(args.steps):
        b, s = oracle_pass(arrays, frac)
        done, secs = done + b, secs + s
    value = done / secs / 1e9
    sample = (f"first {frac:.4%} of every workload of the step (about {done / args.steps / 1e6:.0f} MB per step), "
              "single-threaded C oracle, float64 Kahan / int64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64,i64",
        "data": "synthetic", "config": config_block(),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block():
    return {
        "workload": "rdx suite: fp32 sum+sumsq n=2^24+13 N(0,1) s1; int32->int64 sum n=2^28 U{-2^20..2^20} s2; "
                    "fp32 rowsum 8192x32768 and 1048576x256 U[-1,1) s3; bf16->fp32 sum+sumsq n=2^30+7 N(0,1) s4",
        "bytes_read_per_step": step_bytes(),
        "calls_per_step": len(inputs.SUITE),
        "l2": f"flushed before every timed launch ({FLUSH_BYTES >> 20} MiB write then {FLUSH_BYTES >> 20} MiB read, "
              "untimed)",
    }


# ---------------------------------------------------------------------------
# the GB300 arm
# ---------------------------------------------------------------------------

class Gb300:
    """Device state shared by the GB300 measurements: the step's inputs on the
    device, its seven launches, the L2 flush and the launching stream."""

    def __init__(self, local: int):
        import torch

        from reduction_rdx_sum_gb300 import abi
        from reduction_rdx_sum_gb300.runop import L2Flush

        self.torch, self.abi = torch, abi
        self.dev = torch.device("cuda", local)
        abi.load()
        self.arrays, self.distinct = suite_arrays()
        self.dev_arrays = {}
        for key, host in self.distinct.items():
            t = torch.from_numpy(host.view(np.int16) if host.dtype == np.uint16 else host)
            self.dev_arrays[key] = t.to(self.dev)
        self.ops = []  # (workload, entry point, input, output)
        for w in inputs.SUITE:
            x = self.dev_arrays[self.key(w)]
            if w.op == "rowsum_f32":
                x = x.view(*w.shape)
                out = torch.empty(w.shape[0], dtype=torch.float32, device=self.dev)
                fn = abi.rdx_rowsum_f32
            else:
                out = torch.empty((), dtype=torch.int64 if w.op == "sum_i32" else torch.float32, device=self.dev)
                fn = abi.SCALAR_OPS[w.op]
            self.ops.append((w, fn, x, out))
        self.flush = L2Flush(self.dev, FLUSH_BYTES)
        self.stream = torch.cuda.current_stream(self.dev)

    @staticmethod
    def key(w):
        return (w.dist, w.seed, w.numel)

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def new_outputs(self):
        """A fresh output tensor for each of the step's launches."""
        return [self.torch.full_like(out, -1) for (_, _, _, out) in self.ops]

    def step(self, record=None, outs=None):
        """One pass of the seven launches, each after an (untimed) L2 flush;
        results go to `outs` (default: the launches' own output tensors)."""
        for k, (w, fn, x, out) in enumerate(self.ops):
            self.flush()
            if record is not None:
                record[k][0].record(self.stream)
            fn(x, out=out if outs is None else outs[k], stream=self.stream)
            if record is not None:
                record[k][1].record(self.stream)

    def time_launch(self, fn, iters):
        """Median ms of one flushed launch of fn (two untimed first)."""
        ts = []
        for it in range(iters + 2):
            self.flush()
            e0, e1 = self.event(), self.event()
            e0.record(self.stream)
            fn()
            e1.record(self.stream)
            self.torch.cuda.synchronize()
            if it >= 2:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def time_back_to_back(self, fn, launches=32):
        """ms per launch of fn launched back to back (input left in the L2)."""
        fn()
        self.torch.cuda.synchronize()
        e0, e1 = self.event(), self.event()
        e0.record(self.stream)
        for _ in range(launches):
            fn()
        e1.record(self.stream)
        self.torch.cuda.synchronize()
        return e0.elapsed_time(e1) / launches


def launches_per_step(g: Gb300) -> int:
    """Kernels the step's calls enqueue (the library's own count: one, or two
    where a separate finish kernel follows the tiles)."""
    total = 0
    for (w, _, _, _) in g.ops:
        if w.op == "rowsum_f32":
            total += g.abi.rdx_rowsum_kernels(*w.shape)
        else:
            total += g.abi.rdx_reduce_kernels(w.op, w.numel)
    return total


def figures(ms: float, nbytes: int):
    return {"us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes}


def measure_extras(g: Gb300, per_config, iters):
    """Entry points outside the step, timed the same way."""
    torch, abi, s = g.torch, g.abi, g.stream
    extras = {}
    key2, key5 = g.key(inputs.CFG2_SUM_F32), g.key(inputs.CFG5_SUM_BF16)
    pair = torch.empty(2, dtype=torch.float32, device=g.dev)
    for name, cfg, key, fn in (("c2_sum_sumsq_f32_one_pass", "c2", key2, abi.rdx_sum_sumsq_f32),
                               ("c5_sum_sumsq_bf16_one_pass", "c5", key5, abi.rdx_sum_sumsq_bf16_f32acc)):
        xk = g.dev_arrays[key]
        ms = g.time_launch(lambda: fn(xk, out=pair, stream=s), iters)
        kind = "f32" if "f32" in name else "bf16"
        extras[name] = dict(figures(ms, xk.numel() * xk.element_size()),
                            replaces_us=round(per_config[f"{cfg}_sum_{kind}"]["us"]
                                              + per_config[f"{cfg}_sumsq_{kind}"]["us"], 2))
    # configs that fit in the L2 (config 1: 4 MiB; config 2: 64 MiB): flushed
    # as everywhere else and, labelled as such, with the input L2-resident
    # (back-to-back launches: one launch alone would also time the host)
    small = {w.name: torch.from_numpy(inputs.make(w)).to(g.dev) for w in inputs.SMALL}
    for w in inputs.SMALL + (inputs.CFG2_SUM_F32,):
        xk = small[w.name] if w.name in small else g.dev_arrays[key2]
        outk = torch.empty((), dtype=torch.int64 if w.op == "sum_i32" else torch.float32, device=g.dev)
        fn = abi.SCALAR_OPS[w.op]
        ms = g.time_launch(lambda: fn(xk, out=outk, stream=s), iters)
        hot = g.time_back_to_back(lambda: fn(xk, out=outk, stream=s))
        extras[w.name + ("" if w.name in small else "_l2")] = {
            "us": round(ms * 1e3, 2), "GB/s": round(w.bytes_read / (ms * 1e-3) / 1e9, 1),
            "l2_resident_us": round(hot * 1e3, 2), "l2_resident_GB/s": round(w.bytes_read / (hot * 1e-3) / 1e9, 1)}
    xs = g.dev_arrays[g.key(inputs.CFG4_ROWSUM_WIDE)].view(4, -1)   # 4 rows of 2^26: the split-row path
    rows_out = torch.empty(4, dtype=torch.float32, device=g.dev)
    ms = g.time_launch(lambda: abi.rdx_rowsum_f32(xs, out=rows_out, stream=s), iters)
    extras["rowsum_4x67108864_split"] = figures(ms, 1 << 30)
    # the maximum (the page's atomic_max rule) on the int32 1 GiB array and
    # the fp32 64 MiB array: the same tiled kernel with a max fold
    key3 = g.key(inputs.CFG3_SUM_I32)
    for name, key, fn, dt in (("c3_max_i32", key3, abi.rdx_max_i32, torch.int32),
                              ("c2_max_f32", key2, abi.rdx_max_f32, torch.float32)):
        xk = g.dev_arrays[key]
        om = torch.empty((), dtype=dt, device=g.dev)
        ms = g.time_launch(lambda: fn(xk, out=om, stream=s), iters)
        extras[name] = figures(ms, xk.numel() * xk.element_size())
    # the sum split over 8 GPUs, emulated on this one: each chunk's partial
    # through the one-GPU entry point, then the rank-order combine (9 launches)
    from reduction_rdx_sum_gb300 import shard

    for name, op, key, dt in (("c5_sum_bf16_split8_emulated", "sum_bf16", key5, torch.float32),
                              ("c3_sum_i32_split8_emulated", "sum_i32", key3, torch.int64)):
        xk = g.dev_arrays[key]
        slots = torch.empty(8, dtype=dt, device=g.dev)
        res = torch.empty((), dtype=dt, device=g.dev)
        ms = g.time_launch(lambda: shard.emulate(op, xk, 8, out=res, partials=slots, stream=s), iters)
        extras[name] = dict(figures(ms, xk.numel() * xk.element_size()), launches=9)
    # narrow rows through shared memory: the same 1 GiB viewed as 3 and 12
    # columns (algorithmic bytes: 4 per element read and 4 per row written)
    flat = g.dev_arrays[g.key(inputs.CFG4_ROWSUM_WIDE)].view(-1)
    for cols in (3, 12):
        rows = flat.numel() // cols
        xn = flat[: rows * cols].view(rows, cols)
        on = torch.empty(rows, dtype=torch.float32, device=g.dev)
        ms = g.time_launch(lambda: abi.rdx_rowsum_f32(xn, out=on, stream=s), iters)
        extras[f"rowsum_{rows}x{cols}_narrow"] = dict(figures(ms, rows * cols * 4),
                                                      read_write_GBps=round(rows * (cols + 1) * 4 / (ms * 1e-3) / 1e9, 1))
    return extras


# The step's calls in the order the back-to-back measurement queues them:
# two calls on one array are kept at least L2_APART_BYTES of other reads apart.
BACK_TO_BACK_ORDER = ("c2_sum_f32", "c3_sum_i32", "c5_sum_bf16", "c2_sumsq_f32", "c4_rowsum_8192x32768",
                      "c5_sumsq_bf16", "c4_rowsum_1048576x256")
L2_APART_BYTES = 1 << 30   # well past the GB300's 129 MB L2


def measure_back_to_back(g: Gb300, steps: int):
    """The step's seven calls queued back to back, as a pipeline would run
    them (programmatic dependent launch lets each call start while the one
    before it drains), one L2 flush before each step and two events around
    it.  The two calls on the 64 MiB array (smaller than the L2) are kept
    apart by a 1 GiB and a 2 GiB call, and every other array is larger than
    the L2, so no call finds its input there.  Context for the headline, which
    times every call alone after its own flush."""
    order = list(BACK_TO_BACK_ORDER)
    ops = {w.name: (fn, x, out) for (w, fn, x, out) in g.ops}
    ts = []
    for it in range(steps + 2):
        g.flush()
        e0, e1 = g.event(), g.event()
        e0.record(g.stream)
        for name in order:
            fn, x, out = ops[name]
            fn(x, out=out, stream=g.stream)
        e1.record(g.stream)
        g.torch.cuda.synchronize()
        if it >= 2:
            ts.append(e0.elapsed_time(e1))
    ms = float(np.median(ts))
    return {"GB/s": round(step_bytes() / (ms * 1e-3) / 1e9, 1), "ms_per_step": round(ms, 4), "steps": steps,
            "order": order, "l2": "flushed once before each step; the 64 MiB array's two calls 3 GiB apart"}


def measure_ladder(g: Gb300, launches=5):
    """The page's five block reductions on a float32 input larger than the
    L2 (config 4's 1 GiB of U[-1,1) values, n = 2^28): the partials alone
    (the page's kernel) and the whole sum with the device finish in the same
    launch, each as `launches` back-to-back launches between two events (the
    input streams from HBM every time; many launches put the timer's 2 us
    tick far below the differences between versions).  rdx_sum_f32 on the
    same input, timed the same way, for comparison."""
    torch, abi = g.torch, g.abi
    x = g.dev_arrays[g.key(inputs.CFG4_ROWSUM_WIDE)].view(torch.float32)
    nbytes = x.numel() * 4
    total = torch.empty((), dtype=torch.float32, device=g.dev)
    ladder = {"n": x.numel(), "launches": launches}
    for v in range(1, 6):
        part = torch.empty(abi.rdx_ladder_num_partials(v, x.numel()), dtype=torch.float32, device=g.dev)
        ms = g.time_back_to_back(lambda: abi.rdx_ladder_partials_f32(v, x, out=part, stream=g.stream), launches)
        ms_sum = g.time_back_to_back(lambda: abi.rdx_ladder_sum_f32(v, x, out=total, partials=part, stream=g.stream),
                                     launches)
        ladder[f"v{v}"] = {"us": round(ms * 1e3, 1), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                           "sum_us": round(ms_sum * 1e3, 1), "sum_GB/s": round(nbytes / (ms_sum * 1e-3) / 1e9, 1)}
    ms = g.time_back_to_back(lambda: abi.rdx_sum_f32(x, out=total, stream=g.stream), launches)
    ladder["rdx_sum_f32"] = {"us": round(ms * 1e3, 1), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    return ladder


def measure_sharded(g: Gb300, refs, world, rank, iters, workloads=(inputs.CFG5_SUM_BF16, inputs.CFG3_SUM_I32)):
    """With several ranks: the bf16 sum (2^30 + 7) and the int32 sum (2^28)
    split over the ranks (strong scaling): each rank reduces its chunk, the
    partials are all-gathered over NCCL and combined in rank order.  Time per
    call (L2 flushed before each) is the maximum over ranks; the result must
    match the oracle on every rank."""
    from reduction_rdx_sum_gb300 import shard

    torch = g.torch
    out = {}
    for w in workloads:
        x_local = shard.local_chunk(w.op, g.dev_arrays[g.key(w)], world, rank)
        res = shard.sharded_reduce(w.op, x_local)
        ts = []
        for _ in range(iters):
            g.flush()
            barrier(world)
            e0, e1 = g.event(), g.event()
            e0.record(g.stream)
            res = shard.sharded_reduce(w.op, x_local)
            e1.record(g.stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = max_over_ranks(world, float(np.median(ts)))
        ref, tol = refs[w.name]
        got = res.item()
        ok = got == ref if w.op == "sum_i32" else abs(got - ref) <= tol
        ok = max_over_ranks(world, 0.0 if ok else 1.0) == 0.0
        out[f"{w.name}_split{world}"] = dict(figures(ms, w.bytes_read), scaling="strong", ranks=world, parity_ok=ok)
    return out


def measure_e2e(g: Gb300, per_config, steps, world):
    """The step from pinned host memory.  Every step copies each distinct input
    host -> device on a copy stream, runs the seven launches on the compute
    stream as soon as their input has landed, and copies every result back.
    Arrays go in order of falling compute time, so the reductions of one
    array overlap the copy of the next.  A step's copies wait for the
    previous step's launches (they overwrite the inputs those launches read)."""
    torch, s = g.torch, g.stream
    pinned = {}
    for key, host in g.distinct.items():
        t = torch.empty(host.size, dtype=g.dev_arrays[key].dtype, pin_memory=True)
        t.numpy()[:] = host.view(np.int16) if host.dtype == np.uint16 else host
        pinned[key] = t
    outs_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for (_, _, _, o) in g.ops]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(o.numel() * o.element_size() for (_, _, _, o) in g.ops)
    compute_us = {key: 0.0 for key in g.distinct}
    for (w, _, _, _) in g.ops:
        compute_us[g.key(w)] += per_config[w.name]["us"]
    order = sorted(g.distinct, key=lambda k: -compute_us[k])
    copy_stream = torch.cuda.Stream(g.dev)

    def e2e_step(timeline=None):
        copy_stream.wait_stream(s)
        if timeline is not None:
            timeline["start"] = g.event()
            timeline["start"].record(copy_stream)
        landed = {}
        with torch.cuda.stream(copy_stream):
            for key in order:
                g.dev_arrays[key].copy_(pinned[key], non_blocking=True)
                landed[key] = g.event() if timeline is not None else torch.cuda.Event()
                landed[key].record(copy_stream)
        for key in order:
            s.wait_event(landed[key])
            for (w, fn, x, out) in g.ops:
                if g.key(w) == key:
                    fn(x, out=out, stream=s)
            if timeline is not None:
                timeline[("reduced", key)] = g.event()
                timeline[("reduced", key)].record(s)
        with torch.cuda.stream(s):
            for (_, _, _, out), oh in zip(g.ops, outs_host):
                oh.copy_(out, non_blocking=True)
        if timeline is not None:
            timeline["landed"] = landed
            timeline["end"] = g.event()
            timeline["end"].record(s)

    # one untimed warm-up step, then one untimed step with events after every
    # copy and every array's reductions: where the step's time goes
    e2e_step()
    torch.cuda.synchronize()
    tl = {}
    e2e_step(tl)
    torch.cuda.synchronize()
    t0 = tl["start"]
    timeline, prev = [], 0.0
    for key in order:
        landed_ms = t0.elapsed_time(tl["landed"][key])
        nbytes = pinned[key].numel() * pinned[key].element_size()
        timeline.append({"array": "/".join(w.name for w in inputs.SUITE if g.key(w) == key), "bytes": nbytes,
                         "copy_done_ms": round(landed_ms, 3),
                         "copy_GBps": round(nbytes / max(landed_ms - prev, 1e-6) / 1e6, 1),
                         "reduced_ms": round(t0.elapsed_time(tl[("reduced", key)]), 3)})
        prev = landed_ms
    end_ms = t0.elapsed_time(tl["end"])
    timeline_summary = {"per_array": timeline, "step_ms": round(end_ms, 3),
                        "after_last_copy_ms": round(end_ms - prev, 3)}
    barrier(world)
    ea, eb = g.event(), g.event()
    ea.record(s)
    for _ in range(steps):
        e2e_step()
    eb.record(s)
    torch.cuda.synchronize()
    secs = max_over_ranks(world, ea.elapsed_time(eb) / 1e3)
    return {"value": round(step_bytes() * steps * world / secs / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "h2d_GBps": round(h2d * steps / secs / 1e9, 1), "timeline": timeline_summary}, \
        [oh.numpy().copy() for oh in outs_host]


# ---------------------------------------------------------------------------
# parity of the timed results with the oracle
# ---------------------------------------------------------------------------

TOL_F32, TOL_BF16 = 1e-6, 4e-6   # |gpu - exact| <= tol * sum|term| (+ 1e-30)


def oracle_references(arrays):
    """Oracle value and tolerance of every workload of the step, over the
    whole input: {name: (reference, tolerance)}; integer sums carry
    tolerance 0 (bit-exact)."""
    import oracle

    oracle.build()
    refs = {}
    for w in inputs.SUITE:
        a = arrays[w.name]
        if w.op == "rowsum_f32":
            m = a.reshape(w.shape)
            refs[w.name] = (oracle.rowsum_f32(m), TOL_F32 * oracle.rowabssum_f32(m) + 1e-30)
        elif w.op == "sum_i32":
            refs[w.name] = (oracle.sum_i32(a), 0)
        elif w.op == "sum_f32":
            refs[w.name] = (oracle.sum_f32(a), TOL_F32 * oracle.abssum_f32(a) + 1e-30)
        elif w.op == "sumsq_f32":
            q = oracle.sumsq_f32(a)
            refs[w.name] = (q, TOL_F32 * q + 1e-30)
        elif w.op == "sum_bf16":
            refs[w.name] = (oracle.sum_bf16(a), TOL_BF16 * oracle.abssum_bf16(a) + 1e-30)
        elif w.op == "sumsq_bf16":
            q = oracle.sumsq_bf16(a)
            refs[w.name] = (q, TOL_BF16 * q + 1e-30)
        else:
            raise ValueError(w.op)
    return refs


def parity_report(ops, refs, step_results, label):
    """Compare results with the oracle: per workload the largest
    |result - oracle| / tolerance over its outputs (0 for an exact integer
    sum; any value above 1 fails), and whether every step gave the same
    bits.  step_results: one list of host arrays (one per workload) per
    step, in the order of `ops`."""
    report, ok = {}, True
    for k, (w, _, _, _) in enumerate(ops):
        first = step_results[0][k]
        repeat = all(r[k].tobytes() == first.tobytes() for r in step_results[1:])
        ref, tol = refs[w.name]
        if w.op == "sum_i32":
            exact = int(first.reshape(-1)[0]) == int(ref)
            entry = {"exact": exact, "bitwise_repeat": repeat, "ok": exact and repeat}
        else:
            got = first.astype(np.float64).reshape(-1)
            err = np.abs(got - np.asarray(ref, dtype=np.float64).reshape(-1)) / np.asarray(tol).reshape(-1)
            worst = float(err.max()) if err.size else 0.0
            entry = {"max_err_over_tol": round(worst, 6), "bitwise_repeat": repeat,
                     "ok": bool(np.isfinite(worst) and worst <= 1.0 and repeat)}
        ok = ok and entry["ok"]
        report[w.name] = entry
    report["checked"] = label
    report["ok"] = ok
    return report


def run_gb300(args):
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the library has no CPU path")
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    peak, peak_kind = load_peak()
    g = Gb300(local)

    for _ in range(args.warmup):
        g.step()
    torch.cuda.synchronize()

    # the timed steps: each launch between two events on its stream, each
    # step into outputs of its own (checked against the oracle afterwards)
    events = [[[g.event(), g.event()] for _ in g.ops] for _ in range(args.steps)]
    step_outs = [g.new_outputs() for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(local, os.environ.get("RDX_BENCH_CLOCKS_CSV")) as clk:
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for s in range(args.steps):
            g.step(events[s], step_outs[s])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        barrier(world)
    launch_ms = np.array([[e[0].elapsed_time(e[1]) for e in step] for step in events])  # (steps, ops)
    device_s = max_over_ranks(world, float(launch_ms.sum()) / 1e3)
    value = step_bytes() * args.steps * world / device_s / 1e9

    per_config = {}
    for k, (w, _, _, _) in enumerate(g.ops):
        med = float(np.median(launch_ms[:, k]))
        gbs = w.bytes_read / (med * 1e-3) / 1e9
        per_config[w.name] = {"us": round(med * 1e3, 2), "GB/s": round(gbs, 1),
                              "Gelem/s": round(w.numel / (med * 1e-3) / 1e9, 1),
                              "frac_of_peak": round(gbs / peak, 4), "bytes": w.bytes_read,
                              "ncu_traffic": ncu_traffic(w.name)}
    # roofline of the kernel with the largest share of the step's time
    shares = launch_ms.sum(axis=0) / launch_ms.sum()
    top = int(np.argmax(shares))
    wtop = g.ops[top][0]
    achieved = wtop.bytes_read / (float(launch_ms[:, top].mean()) * 1e-3) / 1e9

    iters = max(3, min(args.steps, 10))
    extras = measure_extras(g, per_config, iters)
    back_to_back = measure_back_to_back(g, iters)
    ladder = measure_ladder(g)
    e2e, e2e_results = measure_e2e(g, per_config, max(1, min(args.steps, 20)), world)

    # parity: every timed step's results and the last end-to-end step's host
    # copies against the oracle over the whole input
    refs = oracle_references(g.arrays)
    timed_results = [[o.cpu().numpy() for o in outs] for outs in step_outs]
    parity = parity_report(g.ops, refs, timed_results,
                           f"all {args.steps} timed steps against the oracle; bitwise equal across them")
    parity_e2e = parity_report(g.ops, refs, [e2e_results], "host copies of the last end-to-end step")
    parity["e2e_ok"] = parity_e2e["ok"]
    if not parity_e2e["ok"]:
        parity["e2e"] = parity_e2e
    sharded = measure_sharded(g, refs, world, rank, iters) if world > 1 else None

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(device_s / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32,i64",
        "data": "synthetic", "config": config_block(),
        "frac_of_peak": round(value / peak, 4),
        "per_config": per_config,
        "roofline": {"bound": "hbm", "kernel": wtop.name, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": ncu_traffic(wtop.name),
                     "algorithmic_bytes_per_launch": wtop.bytes_read, "time_share": round(float(shares[top]), 4),
                     "peak_source": f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": e2e,
        "parity": parity,
        "gpu_launches": launches_per_step(g) * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
        "step_back_to_back": back_to_back,
        "ladder_fp32_n2^28": ladder,
        "extras": extras,
        "kernel_source_hash": kernel_source_hash(),
    }
    if sharded is not None:
        line["sharded"] = sharded
    if rank == 0 and world == 1:
        import oracle

        oracle.build()
        frac = calibrate_oracle(g.arrays, 12.0)
        b, secs, passes = 0, 0.0, 0
        while passes == 0 or (frac >= 1.0 and secs < 10.0 and passes < 4):  # about 10-30 s of oracle work
            pb, ps = oracle_pass(g.arrays, frac)
            b, secs, passes = b + pb, secs + ps, passes + 1
        line["cpu_baseline"] = {
            "value": round(b / secs / 1e9, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {frac:.2%} of every workload of one step, {passes} pass(es) ({b / 1e6:.0f} MB), "
                      f"one thread, {secs:.1f} s"}
        line["cpu_threads"] = cpu_threads_rate(g.arrays)
    ok = parity["ok"] and parity["e2e_ok"] and all(v["parity_ok"] for v in (sharded or {}).values())
    if world > 1:
        ok = max_over_ranks(world, 0.0 if ok else 1.0) == 0.0
    if rank == 0:
        print(json.dumps(line), flush=True)
        if not ok:
            print("bench.py: results differ from the oracle (see \"parity\")", file=sys.stderr, flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0 if ok else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
