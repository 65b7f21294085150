"""Run one reduction entry point on a seeded synthetic input and time it.

For quick timings and for profilers (one kernel, a few launches, a chosen size):

    python -m reduction_rdx_sum_gb300.runop --op sum_bf16 --n 268435456 --iters 3
    python -m reduction_rdx_sum_gb300.runop --op rowsum_f32 --rows 262144 --cols 256
    python -m reduction_rdx_sum_gb300.runop --config c5_sum_bf16     # a workload of the suite
    python -m reduction_rdx_sum_gb300.runop --op rowsum_f32 --rows 16777216 --cols 16 --offset 1
    python -m reduction_rdx_sum_gb300.runop --op rowsum_f32 --rows 2000000 --cols 132 --ld 148   # rows 148 floats apart
    python -m reduction_rdx_sum_gb300.runop --op ladder_partials --version 2 --n 262144 --input page

Before each timed call the L2 is flushed (a write of 512 MiB, then a read of
512 MiB so that no dirty line is left for the timed kernel to write back).
Prints one JSON line per call: microseconds (CUDA events on the launching
stream) and GB/s of input read.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import abi, inputs

OPS = ("sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16", "sum_i32", "rowsum_f32", "sum_f32_noalloc",
       "sum_sumsq_f32", "sum_sumsq_bf16", "max_f32", "max_i32", "bank_probe", "ladder_partials", "ladder_sum")


def make_input(op: str, n: int, rows: int, cols: int, seed: int, dev) -> torch.Tensor:
    if op in ("sum_bf16", "sumsq_bf16", "sum_sumsq_bf16"):
        return torch.from_numpy(inputs.normal_bf16_bits(n, seed).view(np.int16)).to(dev)
    if op in ("sum_i32", "max_i32"):
        return torch.from_numpy(inputs.integers_i32(n, seed, -(1 << 20), 1 << 20)).to(dev)
    if op == "rowsum_f32":
        return torch.from_numpy(inputs.uniform_f32(rows * cols, seed, -1.0, 1.0).reshape(rows, cols)).to(dev)
    return torch.from_numpy(inputs.normal_f32(n, seed)).to(dev)


def entry(op: str, version: int = 5):
    if op == "ladder_partials":
        return lambda x, stream=None: abi.rdx_ladder_partials_f32(version, x, stream=stream)
    if op == "ladder_sum":
        return lambda x, stream=None: abi.rdx_ladder_sum_f32(version, x, stream=stream)
    if op == "rowsum_f32":
        return abi.rdx_rowsum_f32
    if op == "sum_f32_noalloc":
        return abi.rdx_sum_f32_noalloc
    if op in ("sum_sumsq_f32", "sum_sumsq_bf16"):
        return abi.PAIR_OPS[op.split("_")[-1]]
    return abi.SCALAR_OPS[op]


class L2Flush:
    """Evict the L2 without leaving dirty lines: write a buffer larger than the
    L2, then read another one (the read evicts the written lines, paying their
    write-back outside the timed region)."""

    def __init__(self, dev, nbytes: int = 512 << 20):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        return self.r.sum()


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--op", choices=OPS)
    ap.add_argument("--config", choices=[w.name for w in inputs.ALL],
                    help="run one workload of the five configurations (its op, shape and seeded input)")
    ap.add_argument("--n", type=int, default=1 << 28)
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--cols", type=int, default=32768)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--offset", type=int, default=0,
                    help="start the input this many elements into its allocation (a base off 16-byte alignment)")
    ap.add_argument("--ld", type=int, default=None,
                    help="rowsum_f32: rows start every LD floats (a leading dimension >= cols; default cols)")
    ap.add_argument("--version", type=int, default=5, choices=range(1, 6),
                    help="the page's block-reduction version for ladder_partials / ladder_sum")
    ap.add_argument("--input", choices=("seeded", "page"), default="seeded",
                    help="page: the page's own float32 input arange(n) %% 7 (float ops only)")
    args = ap.parse_args(argv)
    if args.offset < 0:
        ap.error("--offset must be >= 0")
    if args.ld is not None and (args.op != "rowsum_f32" or args.ld < args.cols):
        ap.error("--ld applies to --op rowsum_f32 and must be >= --cols")
    if (args.op is None) == (args.config is None):
        ap.error("give exactly one of --op and --config")

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if args.op == "bank_probe":
        # the page's demo 1: cycles per shared load for each of its ten patterns
        for pattern in range(10):
            c = abi.rdx_bank_probe(pattern, iters=max(1, args.iters), device=dev)
            print(json.dumps({"op": "bank_probe", "pattern": pattern, "cycles_per_load": round(c, 2)}), flush=True)
        return 0
    if args.config is not None:
        w = {w.name: w for w in inputs.ALL}[args.config]
        host = inputs.make(w)
        host = host.view(np.int16) if host.dtype == np.uint16 else host
        x = torch.from_numpy(host.reshape(w.shape)).to(dev)
        args.op = w.op
    elif args.input == "page":
        x = torch.from_numpy((np.arange(args.n) % 7).astype(np.float32)).to(dev)
    else:
        x = make_input(args.op, args.n, args.rows, args.cols, args.seed, dev)
    strided = args.ld is not None and args.ld > args.cols
    if strided:  # the same rows, ld floats apart (the gaps zero)
        buf = torch.zeros(args.rows * args.ld + args.offset, dtype=x.dtype, device=dev)
        wide = buf[args.offset:].view(args.rows, args.ld)
        wide[:, :args.cols].copy_(x)
        x = wide[:, :args.cols]
    elif args.offset:
        buf = torch.empty(x.numel() + args.offset, dtype=x.dtype, device=dev)
        x = buf[args.offset:].view(x.shape).copy_(x)
    fn = abi.rdx_rowsum_strided_f32 if strided else entry(args.op, args.version)
    stream = torch.cuda.current_stream(dev)
    flush = None if args.no_flush else L2Flush(dev)
    nbytes = x.numel() * x.element_size()
    for i in range(args.iters):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        out = fn(x, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3
        print(json.dumps({"op": args.op, "iter": i, "us": round(us, 2), "GB/s": round(nbytes / us / 1e3, 1),
                          "bytes": nbytes, "result": out.flatten()[0].item()}), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
