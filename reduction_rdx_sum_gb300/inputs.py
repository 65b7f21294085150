"""Seeded synthetic inputs for the reductions.

This module only draws numbers; it holds none of the reduction arithmetic.  It
is the one piece that the CUDA path's callers (tests, bench) and the CPU oracle
both consume, and it imports neither.

Generator
---------
numpy PCG64, drawn in fixed chunks of ``CHUNK`` = 2^22 elements: chunk ``c`` of
the array for seed ``s`` comes from ``default_rng(SeedSequence([s, c]))``.  The
chunking lets the 2^30-element arrays be filled by several threads while the
values stay independent of the thread count.

Distributions (one per workload):
  * uniform float32 on [lo, hi): ``lo + (hi - lo) * random(float32)``
  * normal(0, 1) float32: ``standard_normal(float32)``
  * uniform integers on [lo, hi] inclusive: ``integers(lo, hi, endpoint=True)``
  * bfloat16: normal(0, 1) float32 rounded to nearest-even on the upper 16 bits
    (the usual float32 -> bfloat16 cast), returned as raw uint16 bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

CHUNK = 1 << 22


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(n: int, dtype, seed: int, draw) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    nchunks = -(-n // CHUNK)

    def job(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, c]))
        draw(rng, out[lo:hi])

    if nchunks <= 1:
        if n:
            job(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(job, range(nchunks)))
    return out


def uniform_f32(n: int, seed: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    """float32 uniform on [lo, hi)."""
    scale = np.float32(hi - lo)
    off = np.float32(lo)

    def draw(rng, dst):
        rng.random(dtype=np.float32, out=dst)
        if scale != 1.0:
            dst *= scale
        if off != 0.0:
            dst += off

    return _fill(n, np.float32, seed, draw)


def normal_f32(n: int, seed: int) -> np.ndarray:
    """float32 normal(0, 1)."""
    return _fill(n, np.float32, seed, lambda rng, dst: rng.standard_normal(dtype=np.float32, out=dst))


def integers_i32(n: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """int32 uniform on the inclusive range [lo, hi]."""
    def draw(rng, dst):
        dst[:] = rng.integers(lo, hi, size=dst.size, endpoint=True, dtype=np.int32)

    return _fill(n, np.int32, seed, draw)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even) and
    return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    step = CHUNK
    for lo in range(0, u.size, step):
        seg = u.reshape(-1)[lo : lo + step].astype(np.uint64)
        lsb = (seg >> 16) & 1
        out.reshape(-1)[lo : lo + step] = ((seg + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return out


def normal_bf16_bits(n: int, seed: int) -> np.ndarray:
    """bfloat16 normal(0, 1) (float32 normal cast to bf16), as uint16 bits."""
    out = np.empty(n, dtype=np.uint16)

    def job(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, c]))
        out[lo:hi] = f32_to_bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))

    nchunks = -(-n // CHUNK)
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(job, range(nchunks)))
    return out


# ---------------------------------------------------------------------------
# The workloads: shapes, value distributions and seeds of the five configurations.
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str          # short key
    op: str            # sum_f32 | sumsq_f32 | sum_i32 | rowsum_f32 | sum_bf16 | sumsq_bf16
    shape: tuple       # (n,) or (rows, cols)
    dist: str          # human-readable recipe
    seed: int

    @property
    def numel(self) -> int:
        p = 1
        for s in self.shape:
            p *= s
        return p

    @property
    def itemsize(self) -> int:
        return {"sum_f32": 4, "sumsq_f32": 4, "sum_i32": 4, "rowsum_f32": 4,
                "sum_bf16": 2, "sumsq_bf16": 2}[self.op]

    @property
    def bytes_read(self) -> int:
        return self.numel * self.itemsize


def make(w: Workload) -> np.ndarray:
    """Materialise a workload's input on the host."""
    n = w.numel
    if w.dist == "U[0,1)":
        a = uniform_f32(n, w.seed, 0.0, 1.0)
    elif w.dist == "U[-1,1)":
        a = uniform_f32(n, w.seed, -1.0, 1.0)
    elif w.dist == "N(0,1)":
        a = normal_f32(n, w.seed)
    elif w.dist == "N(0,1)->bf16":
        a = normal_bf16_bits(n, w.seed)
    elif w.dist.startswith("Z["):
        lo, hi = (int(v) for v in w.dist[2:-1].split(","))
        a = integers_i32(n, w.seed, lo, hi)
    else:
        raise ValueError(f"unknown distribution {w.dist}")
    return a.reshape(w.shape)


# Config 1: the small case (fp32 and int32, n = 2^20).
CFG1_SUM_F32 = Workload("c1_sum_f32", "sum_f32", (1 << 20,), "U[0,1)", 0)
CFG1_SUM_I32 = Workload("c1_sum_i32", "sum_i32", (1 << 20,), "Z[-1000,1000]", 0)
# Config 2: fp32 n = 2^24 + 13 (ragged tail), sum and sum of squares of one array.
CFG2_SUM_F32 = Workload("c2_sum_f32", "sum_f32", ((1 << 24) + 13,), "N(0,1)", 1)
CFG2_SUMSQ_F32 = Workload("c2_sumsq_f32", "sumsq_f32", ((1 << 24) + 13,), "N(0,1)", 1)
# Config 3: int32 n = 2^28 (1 GiB) -> int64.
CFG3_SUM_I32 = Workload("c3_sum_i32", "sum_i32", (1 << 28,), "Z[-1048576,1048576]", 2)
# Config 4: row-segmented fp32, 8192 x 32768 and the skinny 2^20 x 256 (1 GiB each).
CFG4_ROWSUM_WIDE = Workload("c4_rowsum_8192x32768", "rowsum_f32", (8192, 32768), "U[-1,1)", 3)
CFG4_ROWSUM_SKINNY = Workload("c4_rowsum_1048576x256", "rowsum_f32", (1 << 20, 256), "U[-1,1)", 3)
# Config 5: bf16 n = 2^30 + 7 (~2 GiB), fp32 accumulation, sum and sum of squares.
CFG5_SUM_BF16 = Workload("c5_sum_bf16", "sum_bf16", ((1 << 30) + 7,), "N(0,1)->bf16", 4)
CFG5_SUMSQ_BF16 = Workload("c5_sumsq_bf16", "sumsq_bf16", ((1 << 30) + 7,), "N(0,1)->bf16", 4)

SMALL = (CFG1_SUM_F32, CFG1_SUM_I32)
SUITE = (CFG2_SUM_F32, CFG2_SUMSQ_F32, CFG3_SUM_I32, CFG4_ROWSUM_WIDE,
         CFG4_ROWSUM_SKINNY, CFG5_SUM_BF16, CFG5_SUMSQ_BF16)
ALL = SMALL + SUITE
