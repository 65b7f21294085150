"""CPU oracle for the sum reductions.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``reduction_rdx_sum_gb300``) and imports nothing from
it; the two meet only in the seeded input generator, which holds none of the
method's arithmetic.

Contents
--------
``oracle.c`` (loaded here through ctypes)
    The plain definitions, one loop in index order each: float64 Kahan sums for
    float32 and bfloat16 inputs, int64 sums for int32, per-row loops for the
    row-segmented sum, and the maximum by the page's atomic_max rule.  Page
    "03_shared_memory_sync_reduction.py", demo 3: the expected value of every
    reduction version is the float64 sum of the input.
``threads.c`` (a second library, with ``oracle.c`` linked in)
    The multi-core CPU baseline: one contiguous chunk per thread, each run
    through the single-thread loop above, chunk results added in chunk order.
    Not a parity reference; pinned against the single-thread oracle.
``ladder.py``
    The five block-level reduction versions of that page's demo 3, restated in
    numpy float32 in the page's order of operations, giving each block's
    partial sum bit for bit.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, exact rational sums, brute force on tiny inputs and the page's worked
example; none is marked "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_THREADS_SRC = os.path.join(_HERE, "threads.c")
_THREADS_LIB = os.path.join(_HERE, "_liboracle_threads.so")
_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None
_threads_lib = None


def _compile(out: str, srcs: list[str], libs: list[str], force: bool) -> str:
    stale = force or not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(s) for s in srcs)
    if stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, *srcs, "-o", tmp, *libs], check=True)
        os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_liboracle.so`` next to it, and the threaded
    baseline into ``_liboracle_threads.so`` (gcc, no GPU)."""
    _compile(_THREADS_LIB, [_THREADS_SRC, _SRC], ["-lm", "-lpthread"], force)
    return _compile(_LIB, [_SRC], ["-lm"], force)


def use_library(path: str | None) -> None:
    """Load the oracle functions from another build of ``oracle.c`` (the pin
    tests use this to check that planted mistakes are caught); None returns to
    the default build."""
    global _lib
    with _lock:
        _lib = None
    if path is not None:
        _load(path)


def _load(path: str | None = None):
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        p, i64, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
        for name in ("oracle_sum_f32", "oracle_sumsq_f32", "oracle_abssum_f32",
                     "oracle_sum_bf16", "oracle_sumsq_bf16", "oracle_abssum_bf16"):
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = [p, i64], dbl
        lib.oracle_sum_i32.argtypes, lib.oracle_sum_i32.restype = [p, i64], i64
        lib.oracle_sum_i64.argtypes, lib.oracle_sum_i64.restype = [p, i64], i64
        for name in ("oracle_rowsum_f32", "oracle_rowabssum_f32"):
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = [p, i64, i64, p], None
        lib.oracle_max_f32.argtypes, lib.oracle_max_f32.restype = [p, i64], ctypes.c_float
        lib.oracle_max_i32.argtypes, lib.oracle_max_i32.restype = [p, i64], ctypes.c_int32
        _lib = lib
        return lib


def _load_threads():
    global _threads_lib
    with _lock:
        if _threads_lib is None:
            build()
            lib = ctypes.CDLL(_THREADS_LIB)
            p, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_threaded_reduce.argtypes = [c_int, p, i64, c_int, p, p]
            lib.oracle_threaded_reduce.restype = c_int
            lib.oracle_threaded_rowsum_f32.argtypes = [p, i64, i64, c_int, p]
            lib.oracle_threaded_rowsum_f32.restype = c_int
            _threads_lib = lib
        return _threads_lib


def _flat(x: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"oracle expects {np.dtype(dtype)}, got {a.dtype}")
    return a.reshape(-1)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---- float32 -------------------------------------------------------------

def sum_f32(x: np.ndarray) -> float:
    """Sum of float32 values, float64 Kahan, index order."""
    a = _flat(x, np.float32)
    return _load().oracle_sum_f32(_ptr(a), a.size)


def sumsq_f32(x: np.ndarray) -> float:
    """Sum of squares of float32 values (each square exact in float64)."""
    a = _flat(x, np.float32)
    return _load().oracle_sumsq_f32(_ptr(a), a.size)


def abssum_f32(x: np.ndarray) -> float:
    """Sum of |x_i|: the scale of the float32 tolerance."""
    a = _flat(x, np.float32)
    return _load().oracle_abssum_f32(_ptr(a), a.size)


# ---- bfloat16, passed as the raw uint16 bit patterns ----------------------

def sum_bf16(bits: np.ndarray) -> float:
    """Sum of bfloat16 values (given as uint16 bit patterns), each widened exactly."""
    a = _flat(bits, np.uint16)
    return _load().oracle_sum_bf16(_ptr(a), a.size)


def sumsq_bf16(bits: np.ndarray) -> float:
    a = _flat(bits, np.uint16)
    return _load().oracle_sumsq_bf16(_ptr(a), a.size)


def abssum_bf16(bits: np.ndarray) -> float:
    a = _flat(bits, np.uint16)
    return _load().oracle_abssum_bf16(_ptr(a), a.size)


# ---- int32 -> int64 --------------------------------------------------------

def sum_i32(x: np.ndarray) -> int:
    """Exact int64 sum of int32 values."""
    a = _flat(x, np.int32)
    return int(_load().oracle_sum_i32(_ptr(a), a.size))


def sum_i64(x: np.ndarray) -> int:
    """Sum of int64 values modulo 2^64 (as a signed int64): the combine of
    the int64 partials of a sum split into chunks."""
    a = _flat(x, np.int64)
    return int(_load().oracle_sum_i64(_ptr(a), a.size))


# ---- maximum (the page's atomic_max rule, folded from -Inf) ----------------

def max_f32(x: np.ndarray) -> float:
    """Largest float32 value; NaNs are ignored, empty or all-NaN gives -Inf."""
    a = _flat(x, np.float32)
    return float(_load().oracle_max_f32(_ptr(a), a.size))


def max_i32(x: np.ndarray) -> int:
    """Largest int32 value; empty input gives -2^31."""
    a = _flat(x, np.int32)
    return int(_load().oracle_max_i32(_ptr(a), a.size))


# ---- row-segmented float32 -------------------------------------------------

def rowsum_f32(x: np.ndarray) -> np.ndarray:
    """Per-row float64 Kahan sums of a row-major (rows, cols) float32 matrix."""
    a = np.ascontiguousarray(x)
    if a.dtype != np.float32 or a.ndim != 2:
        raise TypeError("rowsum_f32 expects a 2-D float32 array")
    rows, cols = a.shape
    out = np.empty(rows, dtype=np.float64)
    _load().oracle_rowsum_f32(_ptr(a), rows, cols, _ptr(out))
    return out


def rowabssum_f32(x: np.ndarray) -> np.ndarray:
    """Per-row sums of |x|: the per-row tolerance scale."""
    a = np.ascontiguousarray(x)
    if a.dtype != np.float32 or a.ndim != 2:
        raise TypeError("rowabssum_f32 expects a 2-D float32 array")
    rows, cols = a.shape
    out = np.empty(rows, dtype=np.float64)
    _load().oracle_rowabssum_f32(_ptr(a), rows, cols, _ptr(out))
    return out


# ---- the multi-core baseline (threads.c) ------------------------------------

_THREADED_OPS = {"sum_f32": (0, np.float32), "sumsq_f32": (1, np.float32), "sum_bf16": (2, np.uint16),
                 "sumsq_bf16": (3, np.uint16), "sum_i32": (4, np.int32)}


def default_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def threaded(op: str, x: np.ndarray, threads: int | None = None):
    """``op`` (one of sum_f32, sumsq_f32, sum_bf16, sumsq_bf16, sum_i32) on
    ``threads`` host threads, one contiguous chunk each; float for the float
    ops, int for sum_i32."""
    code, dtype = _THREADED_OPS[op]
    a = _flat(x, dtype)
    d, i = ctypes.c_double(0.0), ctypes.c_int64(0)
    rc = _load_threads().oracle_threaded_reduce(code, _ptr(a), a.size, int(threads or default_threads()),
                                                ctypes.byref(d), ctypes.byref(i))
    if rc != 0:
        raise RuntimeError(f"oracle_threaded_reduce({op}) failed")
    return int(i.value) if op == "sum_i32" else float(d.value)


def threaded_rowsum_f32(x: np.ndarray, threads: int | None = None) -> np.ndarray:
    """Per-row sums with the rows split over ``threads`` host threads."""
    a = np.ascontiguousarray(x)
    if a.dtype != np.float32 or a.ndim != 2:
        raise TypeError("threaded_rowsum_f32 expects a 2-D float32 array")
    rows, cols = a.shape
    out = np.empty(rows, dtype=np.float64)
    if _load_threads().oracle_threaded_rowsum_f32(_ptr(a), rows, cols, int(threads or default_threads()),
                                                  _ptr(out)) != 0:
        raise RuntimeError("oracle_threaded_rowsum_f32 failed")
    return out


from .ladder import LADDER_BLOCK, ladder_partials, ladder_segment, VERSIONS  # noqa: E402,F401
