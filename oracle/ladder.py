"""The five block-level sum reductions of the page
"03_shared_memory_sync_reduction.py", demo 3 (parallel reduction, after
Harris, "Optimizing Parallel Reduction in CUDA", 2007), restated in numpy.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see ``oracle/__init__.py``).

Each version maps the input to one float32 partial sum per block; a block of
B threads covers B consecutive inputs (versions 1-3) or 2B (versions 4-5).
Every step below is the page's step, applied to all blocks at once: a row of
the (blocks, B) array is one block's shared-memory buffer ``sdata``, and each
``a + b`` is the same float32 addition a thread performs, on the same two
operands, so the partials are exact to the bit.  All float32 arithmetic
rounds to nearest, as the GPU's ``add.rn.f32`` does.

Where the page is silent: it launches ``n // (B * per_thread)`` blocks and
reads no index past the end (it requires divisible n).  The reading taken here
is the masking convention of the page "simt_lab.py" (kernels mask ``i < n``):
the last block is partial and an input past the end counts as 0.  Adding a
0.0 changes no finite value, so divisible inputs are unaffected.
"""
from __future__ import annotations

import numpy as np

LADDER_BLOCK = 256  # the page's block size B for demo 3


def ladder_segment(version: int, block: int = LADDER_BLOCK) -> int:
    """Inputs covered by one block: B for versions 1-3, 2B for 4-5."""
    if version not in VERSIONS:
        raise ValueError(f"version must be 1..5, got {version}")
    return block if version <= 3 else 2 * block


def _blocks(x: np.ndarray, seg: int) -> np.ndarray:
    """(blocks, seg) float32 view of x, the missing tail filled with 0."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    nb = -(-x.size // seg)
    buf = np.zeros(nb * seg, dtype=np.float32)
    buf[: x.size] = x
    return buf.reshape(nb, seg)


def _sequential_tail(sdata: np.ndarray, block: int, stop_at: int = 1) -> None:
    """Sequential addressing: for s = B/2, B/4, ..., stop_at the first s threads
    do sdata[tid] += sdata[tid + s] (page: ``_sequential_tail``)."""
    s = block // 2
    while s >= stop_at:
        sdata[:, :s] = sdata[:, :s] + sdata[:, s : 2 * s]
        s //= 2


def v1_interleaved_divergent(x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Version 1: at step s = 1, 2, 4, ... the threads whose tid is a multiple
    of 2s add sdata[tid + s] into sdata[tid]; thread 0 writes sdata[0]."""
    sdata = _blocks(x, block).copy()
    s = 1
    while s < block:
        tid = np.arange(0, block, 2 * s)  # the threads with tid % (2s) == 0
        sdata[:, tid] = sdata[:, tid] + sdata[:, tid + s]
        s *= 2
    return sdata[:, 0].copy()


def v2_interleaved_strided(x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Version 2: at step s thread tid works on index = 2*s*tid (if < B):
    sdata[index] += sdata[index + s].  Same operand pairs as version 1,
    assigned to consecutive threads."""
    sdata = _blocks(x, block).copy()
    s = 1
    while s < block:
        index = 2 * s * np.arange(block)
        index = index[index < block]
        sdata[:, index] = sdata[:, index] + sdata[:, index + s]
        s *= 2
    return sdata[:, 0].copy()


def v3_sequential(x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Version 3: load one input per thread, then the sequential-addressing
    loop down to s = 1."""
    sdata = _blocks(x, block).copy()
    _sequential_tail(sdata, block)
    return sdata[:, 0].copy()


def v4_first_add(x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Version 4: each block covers 2B inputs; thread tid first adds
    in[i] + in[i + B] (i = bx*2B + tid), then the sequential loop."""
    seg = _blocks(x, 2 * block)
    sdata = seg[:, :block] + seg[:, block:]
    _sequential_tail(sdata, block)
    return sdata[:, 0].copy()


def v5_warp_shuffle(x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Version 5: version 4's load, the sequential loop stopped at s = 64, then
    warp 0 forms val = sdata[tid] + sdata[tid + 32] and five shuffle-down
    steps (offsets 16, 8, 4, 2, 1): lane l adds the value of lane l + offset,
    or its own value when l + offset falls outside the warp."""
    if block < 64:
        raise ValueError("version 5 needs B >= 64")
    seg = _blocks(x, 2 * block)
    sdata = seg[:, :block] + seg[:, block:]
    _sequential_tail(sdata, block, stop_at=64)
    val = sdata[:, 0:32] + sdata[:, 32:64]
    for off in (16, 8, 4, 2, 1):
        received = val.copy()  # lanes past the warp's end get their own value
        received[:, : 32 - off] = val[:, off:32]
        val = val + received
    return val[:, 0].copy()


VERSIONS = {
    1: v1_interleaved_divergent,
    2: v2_interleaved_strided,
    3: v3_sequential,
    4: v4_first_add,
    5: v5_warp_shuffle,
}


def ladder_partials(version: int, x: np.ndarray, block: int = LADDER_BLOCK) -> np.ndarray:
    """Per-block float32 partial sums of ``version`` (1..5) over x."""
    if version not in VERSIONS:
        raise ValueError(f"version must be 1..5, got {version}")
    if block & (block - 1) or block < 2:
        raise ValueError("block size must be a power of two")
    if np.asarray(x).size == 0:
        return np.zeros(0, dtype=np.float32)
    return VERSIONS[version](x, block)
