"""Python binding of librdx.so: the C-ABI entry points under the same names.

Argument marshalling only: each function checks the tensors it is given,
passes their device pointers, sizes and the current CUDA stream to the C
entry point, and raises ``RdxError`` on a non-zero status.  All arithmetic
happens in the CUDA kernels.  If the library has not been built (see
``reduction_rdx_sum_gb300.build``), every call raises; there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from .build import LIB

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rdx.h")

RDX_OK = 0
RDX_ERR_INVALID_ARG = 1
RDX_ERR_CUDA = 2
RDX_ERR_ALLOC = 3
RDX_ERR_UNSUPPORTED_DEVICE = 4

_lock = threading.Lock()
_lib = None


class RdxError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})" + (f": {detail}" if detail else ""))
        self.status = status


def declared_symbols() -> list[str]:
    """Names of the functions include/rdx.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rdx_[a-z0-9_]+)\s*\(", text)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Open librdx.so (once) and declare the C signatures.  RDX_LIBRARY may
    name another build of it (the checked build, for instance)."""
    global _lib
    path = path or os.environ.get("RDX_LIBRARY") or LIB
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is not built; run reduction_rdx_sum_gb300.build.build() "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("rdx_sum_f32", "rdx_sumsq_f32", "rdx_sum_bf16_f32acc", "rdx_sumsq_bf16_f32acc",
                     "rdx_sum_i32_i64", "rdx_sum_sumsq_f32", "rdx_sum_sumsq_bf16_f32acc", "rdx_max_f32",
                     "rdx_max_i32", "rdx_sum_f32_noalloc"):
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = [vp, i64, vp, vp], i32
        lib.rdx_rowsum_f32.argtypes, lib.rdx_rowsum_f32.restype = [vp, i64, i64, vp, vp], i32
        lib.rdx_rowsum_strided_f32.argtypes = [vp, i64, i64, i64, vp, vp]
        lib.rdx_rowsum_strided_f32.restype = i32
        lib.rdx_workspace_bytes.argtypes, lib.rdx_workspace_bytes.restype = [], ctypes.c_size_t
        lib.rdx_reduce_kernels.argtypes, lib.rdx_reduce_kernels.restype = [i32, i64], i32
        lib.rdx_rowsum_kernels.argtypes, lib.rdx_rowsum_kernels.restype = [i64, i64], i32
        lib.rdx_reduce_ws.argtypes = [i32, vp, i64, vp, vp, ctypes.c_size_t, vp]
        lib.rdx_reduce_ws.restype = i32
        lib.rdx_bank_probe.argtypes, lib.rdx_bank_probe.restype = [i32, i32, vp, vp, vp], i32
        lib.rdx_bank_probe_loads_per_iter.argtypes, lib.rdx_bank_probe_loads_per_iter.restype = [], i32
        lib.rdx_debug_build.argtypes, lib.rdx_debug_build.restype = [], i32
        lib.rdx_debug_violations.argtypes, lib.rdx_debug_violations.restype = [vp, i32], i32
        lib.rdx_wait_timeouts.argtypes, lib.rdx_wait_timeouts.restype = [vp, i32], i32
        lib.rdx_debug_stage_timeout.argtypes, lib.rdx_debug_stage_timeout.restype = [vp, i64, i64, vp, vp], i32
        lib.rdx_ladder_partials_f32.argtypes = [i32, vp, i64, vp, vp]
        lib.rdx_ladder_partials_f32.restype = i32
        lib.rdx_ladder_num_partials.argtypes, lib.rdx_ladder_num_partials.restype = [i32, i64], i64
        lib.rdx_ladder_sum_f32.argtypes, lib.rdx_ladder_sum_f32.restype = [i32, vp, i64, vp, vp, vp], i32
        lib.rdx_shard_range.argtypes = [i64, i32, i32, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.rdx_shard_range.restype = i32
        lib.rdx_combine_max_parts.argtypes, lib.rdx_combine_max_parts.restype = [], i32
        for name in ("rdx_combine_f32", "rdx_combine_f32x2", "rdx_combine_i64"):
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = [vp, i32, vp, vp], i32
        lib.rdx_status_string.argtypes, lib.rdx_status_string.restype = [i32], ctypes.c_char_p
        lib.rdx_last_cuda_error.argtypes, lib.rdx_last_cuda_error.restype = [], ctypes.c_char_p
        lib.rdx_shutdown.argtypes, lib.rdx_shutdown.restype = [], None
        lib.rdx_release_stream.argtypes, lib.rdx_release_stream.restype = [vp], i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().rdx_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != RDX_OK:
        raise RdxError(fn, status, load().rdx_last_cuda_error().decode())


try:  # the current stream's cudaStream_t by device index, without building a Stream object
    _current_raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover - builds without the accessor
    def _current_raw_stream(index: int) -> int:
        return int(torch.cuda.current_stream(index).cuda_stream)


def _launch(fn, device, stream, *args) -> int:
    """fn(*args, stream handle) with `device` current: the C entry points
    launch on the current device, in `stream` (default: the current stream
    of `device`).  The device is switched only when it is not current."""
    index = device.index if isinstance(device, torch.device) else int(device)
    if index == torch.cuda.current_device():
        return fn(*args, _current_raw_stream(index) if stream is None else int(stream.cuda_stream))
    with torch.cuda.device(index):
        return fn(*args, _current_raw_stream(index) if stream is None else int(stream.cuda_stream))


def _input(x: torch.Tensor, dtypes, what: str) -> torch.Tensor:
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError(f"{what}: expected a CUDA tensor")
    if x.dtype not in dtypes:
        raise TypeError(f"{what}: expected dtype in {dtypes}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    return x


def _output(out, like: torch.Tensor, dtype, shape) -> torch.Tensor:
    if out is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    if not out.is_cuda or out.dtype != dtype or tuple(out.shape) != tuple(shape) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous CUDA {dtype} tensor of shape {tuple(shape)}")
    return out


def _scalar(name: str, x: torch.Tensor, dtypes, out_dtype, out, stream, shape=()) -> torch.Tensor:
    lib = load()
    x = _input(x, dtypes, name)
    out = _output(out, x, out_dtype, shape)
    st = _launch(getattr(lib, name), x.device, stream, x.data_ptr(), x.numel(), out.data_ptr())
    _check(name, st)
    return out


_BF16 = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else (torch.bfloat16, torch.int16)


def rdx_sum_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of a float32 tensor."""
    return _scalar("rdx_sum_f32", x, (torch.float32,), torch.float32, out, stream)


def rdx_sumsq_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of squares of a float32 tensor."""
    return _scalar("rdx_sumsq_f32", x, (torch.float32,), torch.float32, out, stream)


def rdx_sum_bf16_f32acc(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of a bfloat16 tensor (or its raw 16-bit patterns)."""
    return _scalar("rdx_sum_bf16_f32acc", x, _BF16, torch.float32, out, stream)


def rdx_sumsq_bf16_f32acc(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of squares of a bfloat16 tensor."""
    return _scalar("rdx_sumsq_bf16_f32acc", x, _BF16, torch.float32, out, stream)


def rdx_sum_i32_i64(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d int64 tensor: the exact sum of an int32 tensor."""
    return _scalar("rdx_sum_i32_i64", x, (torch.int32,), torch.int64, out, stream)


def rdx_sum_sumsq_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """(2,) float32 tensor [sum, sum of squares] of a float32 tensor, one pass."""
    return _scalar("rdx_sum_sumsq_f32", x, (torch.float32,), torch.float32, out, stream, shape=(2,))


def rdx_sum_sumsq_bf16_f32acc(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """(2,) float32 tensor [sum, sum of squares] of a bfloat16 tensor, one pass."""
    return _scalar("rdx_sum_sumsq_bf16_f32acc", x, _BF16, torch.float32, out, stream, shape=(2,))


def rdx_max_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the maximum of a float32 tensor (NaNs skipped; empty gives -Inf)."""
    return _scalar("rdx_max_f32", x, (torch.float32,), torch.float32, out, stream)


def rdx_max_i32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d int32 tensor: the maximum of an int32 tensor (empty gives -2^31)."""
    return _scalar("rdx_max_i32", x, (torch.int32,), torch.int32, out, stream)


def rdx_rowsum_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """(rows,) float32 tensor: per-row sums of a contiguous 2-D float32 tensor."""
    lib = load()
    x = _input(x, (torch.float32,), "rdx_rowsum_f32")
    if x.dim() != 2:
        raise ValueError("rdx_rowsum_f32: expected a 2-D tensor")
    rows, cols = x.shape
    out = _output(out, x, torch.float32, (rows,))
    st = _launch(lib.rdx_rowsum_f32, x.device, stream, x.data_ptr(), rows, cols, out.data_ptr())
    _check("rdx_rowsum_f32", st)
    return out


def rdx_rowsum_strided_f32(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """(rows,) float32 tensor: per-row sums of a 2-D float32 tensor whose rows
    are contiguous (stride(1) == 1) and start every stride(0) elements, such
    as a column slice of a wider matrix."""
    lib = load()
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32 or x.dim() != 2:
        raise TypeError("rdx_rowsum_strided_f32: expected a 2-D float32 CUDA tensor")
    rows, cols = x.shape
    if cols > 1 and x.stride(1) != 1:
        raise ValueError("rdx_rowsum_strided_f32: rows must be contiguous (stride(1) == 1)")
    ld = x.stride(0) if rows > 1 else cols
    out = _output(out, x, torch.float32, (rows,))
    st = _launch(lib.rdx_rowsum_strided_f32, x.device, stream, x.data_ptr(), rows, cols, ld, out.data_ptr())
    _check("rdx_rowsum_strided_f32", st)
    return out


# RDX_OP_* codes of include/rdx.h, by operation name.
OP_CODES = {"sum_f32": 0, "sumsq_f32": 1, "sum_bf16": 2, "sumsq_bf16": 3, "sum_i32": 4,
            "sum_sumsq_f32": 5, "sum_sumsq_bf16": 6, "max_f32": 7, "max_i32": 8}
_OP_IN = {0: (torch.float32,), 1: (torch.float32,), 2: _BF16, 3: _BF16, 4: (torch.int32,), 5: (torch.float32,),
          6: _BF16, 7: (torch.float32,), 8: (torch.int32,)}
_OP_OUT = {0: (torch.float32, ()), 1: (torch.float32, ()), 2: (torch.float32, ()), 3: (torch.float32, ()),
           4: (torch.int64, ()), 5: (torch.float32, (2,)), 6: (torch.float32, (2,)), 7: (torch.float32, ()),
           8: (torch.int32, ())}


def rdx_workspace_bytes() -> int:
    return int(load().rdx_workspace_bytes())


def rdx_reduce_kernels(op, n: int) -> int:
    """Kernels one call of scalar reduction ``op`` (name or RDX_OP_* code) on n elements enqueues."""
    return int(load().rdx_reduce_kernels(OP_CODES[op] if isinstance(op, str) else int(op), n))


def rdx_rowsum_kernels(rows: int, cols: int) -> int:
    """Kernels one rdx_rowsum_f32 call on a rows x cols matrix enqueues."""
    return int(load().rdx_rowsum_kernels(rows, cols))


def rdx_reduce_ws(op, x: torch.Tensor, workspace: torch.Tensor, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Scalar reduction ``op`` (a name of OP_CODES or an RDX_OP_* code) with a
    caller-owned workspace (a CUDA tensor of at least rdx_workspace_bytes()
    bytes, zero-filled before its first use)."""
    lib = load()
    code = OP_CODES[op] if isinstance(op, str) else int(op)
    if code not in _OP_IN:
        raise ValueError(f"rdx_reduce_ws: unknown op {op}")
    x = _input(x, _OP_IN[code], "rdx_reduce_ws")
    dt, shape = _OP_OUT[code]
    out = _output(out, x, dt, shape)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("rdx_reduce_ws: workspace must be a contiguous CUDA tensor")
    st = _launch(lib.rdx_reduce_ws, x.device, stream, code, x.data_ptr(), x.numel(), out.data_ptr(),
                 workspace.data_ptr(), workspace.numel() * workspace.element_size())
    _check("rdx_reduce_ws", st)
    return out


def rdx_bank_probe(pattern: int, iters: int = 256, device=None, stream=None) -> float:
    """Clock cycles per shared-memory load instruction of the page's bank
    pattern ``pattern`` (0..9), measured by one warp on the GPU."""
    lib = load()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    cycles = torch.zeros(1, dtype=torch.int64, device=device)
    sink = torch.zeros(32, dtype=torch.int32, device=device)
    st = _launch(lib.rdx_bank_probe, device, stream, pattern, iters, cycles.data_ptr(), sink.data_ptr())
    _check("rdx_bank_probe", st)
    return cycles.item() / (iters * lib.rdx_bank_probe_loads_per_iter())


def rdx_ladder_num_partials(version: int, n: int) -> int:
    return int(load().rdx_ladder_num_partials(version, n))


def rdx_ladder_partials_f32(version: int, x: torch.Tensor, out: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Per-block partials of the page's block-reduction ``version`` (1..5)."""
    lib = load()
    x = _input(x, (torch.float32,), "rdx_ladder_partials_f32")
    nb = lib.rdx_ladder_num_partials(version, x.numel())
    if nb < 0:
        raise ValueError(f"rdx_ladder_partials_f32: bad version {version}")
    out = _output(out, x, torch.float32, (nb,))
    st = _launch(lib.rdx_ladder_partials_f32, x.device, stream, version, x.data_ptr(), x.numel(), out.data_ptr())
    _check("rdx_ladder_partials_f32", st)
    return out


def rdx_sum_f32_noalloc(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of a float32 tensor, computed with the
    library's static scratch instead of an allocated workspace (for callers
    that may not allocate device memory; calls must not overlap on the GPU)."""
    return _scalar("rdx_sum_f32_noalloc", x, (torch.float32,), torch.float32, out, stream)


def rdx_ladder_sum_f32(version: int, x: torch.Tensor, out: torch.Tensor | None = None,
                       partials: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the sum of a float32 tensor by the page's block
    reduction ``version`` (1..5), its per-block partials (left in
    ``partials``) added on the device in the same launch."""
    lib = load()
    x = _input(x, (torch.float32,), "rdx_ladder_sum_f32")
    nb = lib.rdx_ladder_num_partials(version, x.numel())
    if nb < 0:
        raise ValueError(f"rdx_ladder_sum_f32: bad version {version}")
    partials = _output(partials, x, torch.float32, (nb,))
    out = _output(out, x, torch.float32, ())
    st = _launch(lib.rdx_ladder_sum_f32, x.device, stream, version, x.data_ptr(), x.numel(), partials.data_ptr(),
                 out.data_ptr())
    _check("rdx_ladder_sum_f32", st)
    return out


def rdx_shard_range(n: int, parts: int, rank: int, granule: int) -> tuple[int, int]:
    """(lo, hi): the chunk of rank ``rank`` among ``parts`` sharing ``n``
    elements cut in whole granules of ``granule`` elements (host only)."""
    lo, hi = ctypes.c_int64(0), ctypes.c_int64(0)
    _check("rdx_shard_range", load().rdx_shard_range(n, parts, rank, granule, ctypes.byref(lo), ctypes.byref(hi)))
    return int(lo.value), int(hi.value)


def rdx_combine_max_parts() -> int:
    return int(load().rdx_combine_max_parts())


def _combine(name: str, parts: torch.Tensor, dtype, width: int, out, stream) -> torch.Tensor:
    lib = load()
    parts = _input(parts, (dtype,), name)
    if parts.numel() % width:
        raise ValueError(f"{name}: expected {width} values per partial")
    p = parts.numel() // width
    out = _output(out, parts, dtype, () if width == 1 else (width,))
    st = _launch(getattr(lib, name), parts.device, stream, parts.data_ptr(), p, out.data_ptr())
    _check(name, st)
    return out


def rdx_combine_f32(parts: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d float32 tensor: the float32 partials ``parts`` added in index (rank) order."""
    return _combine("rdx_combine_f32", parts, torch.float32, 1, out, stream)


def rdx_combine_f32x2(parts: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """(2,) float32 tensor: the [sum, sum of squares] pairs ``parts`` (p x 2)
    added component-wise in rank order."""
    return _combine("rdx_combine_f32x2", parts, torch.float32, 2, out, stream)


def rdx_combine_i64(parts: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """0-d int64 tensor: the int64 partials ``parts`` added (modulo 2^64)."""
    return _combine("rdx_combine_i64", parts, torch.int64, 1, out, stream)


def rdx_shutdown() -> None:
    load().rdx_shutdown()


def rdx_release_stream(stream=None, device=None) -> bool:
    """Free the library's workspace for ``stream`` (default: the current
    stream) on ``device`` (default: the current device); True if one was
    freed.  Call after the stream's work has completed."""
    index = torch.cuda.current_device() if device is None else torch.device(device).index
    with torch.cuda.device(index):
        handle = _current_raw_stream(index) if stream is None else int(stream.cuda_stream)
        return bool(load().rdx_release_stream(handle))


def rdx_debug_build() -> bool:
    """True when the loaded library is the checked build (RDX_DEBUG=1)."""
    return bool(load().rdx_debug_build())


def rdx_debug_violations(reset: bool = False) -> int:
    """Out-of-range accesses the checked build caught (0 in a normal build)."""
    count = ctypes.c_uint64(0)
    _check("rdx_debug_violations", load().rdx_debug_violations(ctypes.byref(count), int(reset)))
    return int(count.value)


def rdx_wait_timeouts(reset: bool = False) -> int:
    """Staging waits of the narrow-row kernel that gave up on the current
    device since the last reset (synchronizes the device)."""
    count = ctypes.c_uint64(0)
    _check("rdx_wait_timeouts", load().rdx_wait_timeouts(ctypes.byref(count), int(reset)))
    return int(count.value)


def rdx_debug_stage_timeout(x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Test hook: one narrow-row tile of the 2-D float32 tensor x (rows *
    cols <= 6144) whose staging wait cannot complete, so that it gives up
    after one second; out (rows float32 values) is left unwritten."""
    if x.dim() != 2 or x.dtype != torch.float32 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous 2-D float32 CUDA tensor")
    rows, cols = x.shape
    _check("rdx_debug_stage_timeout",
           _launch(load().rdx_debug_stage_timeout, x.device, stream, x.data_ptr(), rows, cols, out.data_ptr()))


# Entry points by operation name, for the tests and the bench.
SCALAR_OPS = {
    "sum_f32": rdx_sum_f32,
    "sumsq_f32": rdx_sumsq_f32,
    "sum_bf16": rdx_sum_bf16_f32acc,
    "sumsq_bf16": rdx_sumsq_bf16_f32acc,
    "sum_i32": rdx_sum_i32_i64,
    "max_f32": rdx_max_f32,
    "max_i32": rdx_max_i32,
}

# One-pass [sum, sum of squares] entry points by input type.
PAIR_OPS = {
    "f32": rdx_sum_sumsq_f32,
    "bf16": rdx_sum_sumsq_bf16_f32acc,
}
