"""The checked build (RDX_DEBUG=1) on the GPU: the parity cases run through a
library whose kernels test every global load and store against its buffer.
Results must still match the oracle and no access may fall outside.  (The
checked build skips an out-of-range access instead of performing it, so this
runs no risk of a fault; it stands in for a memory sanitizer.)"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, build, inputs

from test_parity_gpu import DEV, VEC, check, host_input, to_device

pytestmark = pytest.mark.gpu

CHECKED = os.path.join(os.path.dirname(build.LIB), "..", "_build", "librdx_checked.so")
CODES = abi.OP_CODES
OUT = {"sum_i32": torch.int64, "max_i32": torch.int32}


@pytest.fixture(scope="module")
def lib():
    path = build.build(defines=["-DRDX_DEBUG=1"], out=os.path.abspath(CHECKED))
    oracle.build()
    torch.cuda.set_device(DEV)
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.rdx_reduce_ws.argtypes = [i32, vp, i64, vp, vp, ctypes.c_size_t, vp]
    lib.rdx_rowsum_strided_f32.argtypes = [vp, i64, i64, i64, vp, vp]
    lib.rdx_ladder_partials_f32.argtypes = [i32, vp, i64, vp, vp]
    lib.rdx_ladder_num_partials.argtypes, lib.rdx_ladder_num_partials.restype = [i32, i64], i64
    lib.rdx_ladder_sum_f32.argtypes = [i32, vp, i64, vp, vp, vp]
    lib.rdx_debug_violations.argtypes = [vp, i32]
    lib.rdx_workspace_bytes.restype = ctypes.c_size_t
    for name in ("rdx_sum_f32", "rdx_sum_i32_i64", "rdx_max_f32"):
        getattr(lib, name).argtypes = [vp, i64, vp, vp]
    assert lib.rdx_debug_build() == 1
    count = ctypes.c_uint64(0)
    assert lib.rdx_debug_violations(ctypes.byref(count), 1) == 0
    return lib


def violations(lib):
    count = ctypes.c_uint64(99)
    assert lib.rdx_debug_violations(ctypes.byref(count), 0) == 0
    return count.value


def stream():
    return torch.cuda.current_stream(DEV).cuda_stream


@pytest.mark.parametrize("op", ["sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16", "sum_i32", "max_f32", "max_i32",
                                "sum_sumsq_f32", "sum_sumsq_bf16"])
def test_scalar_ops_stay_in_bounds(lib, op):
    ws = torch.zeros(lib.rdx_workspace_bytes(), dtype=torch.uint8, device=DEV)
    src = {"max_f32": "sum_f32", "max_i32": "sum_i32", "sum_sumsq_f32": "sum_f32",
           "sum_sumsq_bf16": "sum_bf16"}.get(op, op)
    for n in (0, 1, 3, 7, 8, 9, 33, 257, 4097, 65537, (1 << 20) + 3, (1 << 24) + 13):
        host = host_input(src, n, seed=n % 41)
        for offset in range(0, VEC[src], 3):
            x = to_device(host, offset)
            shape = (2,) if op.startswith("sum_sumsq") else ()
            out = torch.empty(shape, dtype=OUT.get(op, torch.float32), device=DEV)
            assert lib.rdx_reduce_ws(CODES[op], x.data_ptr(), n, out.data_ptr(), ws.data_ptr(), ws.numel(),
                                     stream()) == 0
            torch.cuda.synchronize()
            if op.startswith("max"):
                ref = oracle.max_f32(host) if op == "max_f32" else oracle.max_i32(host)
                assert out.item() == ref
            elif op.startswith("sum_sumsq"):
                s_op, q_op = ("sum_f32", "sumsq_f32") if op.endswith("f32") else ("sum_bf16", "sumsq_bf16")
                check(s_op, host, out[0].item())
                check(q_op, host, out[1].item())
            else:
                check(op, host, out.item())
    assert violations(lib) == 0


def test_library_workspace_path_stays_in_bounds(lib):
    for n in (1 << 20, (1 << 22) + 1):
        host = host_input("sum_f32", n, seed=3)
        x = to_device(host, 1)
        out = torch.empty((), device=DEV)
        assert lib.rdx_sum_f32(x.data_ptr(), n, out.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        check("sum_f32", host, out.item())
    assert violations(lib) == 0


ROWS = [(1, 1, 1), (3, 5, 5), (7, 3, 8), (33, 255, 257), (1000, 256, 256), (100, 256, 300), (64, 1023, 1025),
        (17, 4099, 4099), (8, 100_000, 100_003), (2, 1 << 20, (1 << 20) + 1), (4, 16384, 16384), (50_000, 7, 7),
        (40, 5121, 5121), (20, 6001, 6007), (2100, 16385, 16385)]


@pytest.mark.parametrize("shape", ROWS, ids=str)
def test_row_sums_stay_in_bounds(lib, shape):
    rows, cols, ld = shape
    full = inputs.uniform_f32(rows * ld, seed=rows + cols, lo=-1.0, hi=1.0).reshape(rows, ld)
    for start in (0, 1):
        if start + cols > ld and rows > 1:
            continue
        x = torch.from_numpy(full).to(DEV)
        out = torch.empty(rows, device=DEV)
        c = min(cols, ld - start)
        assert lib.rdx_rowsum_strided_f32(x.data_ptr() + 4 * start, rows, c, ld, out.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        host = np.ascontiguousarray(full[:, start:start + c])
        tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
        assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)
    assert violations(lib) == 0


@pytest.mark.parametrize("cols", [1, 2, 3, 4, 6, 8, 12, 16, 20, 31, 32, 40, 50, 52, 56, 63, 64])
def test_narrow_row_sums_stay_in_bounds(lib, cols):
    # contiguous rows of at most 64 columns: tiles of whole rows staged in
    # shared memory, at every 4-byte misalignment of the base (the rotated and
    # aligned-down reads of unaligned 8, 12, 16, ... columns and the bulk-copy
    # staging included)
    rows = 3 * (6144 // cols) + 5
    host = inputs.uniform_f32(rows * cols, seed=cols, lo=-1.0, hi=1.0).reshape(rows, cols)
    for offset in range(4):
        x = to_device(host.reshape(-1), offset)
        out = torch.empty(rows, device=DEV)
        assert lib.rdx_rowsum_strided_f32(x.data_ptr(), rows, cols, cols, out.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
        assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)
    assert violations(lib) == 0


@pytest.mark.parametrize("cols", [68, 92, 132, 184, 260, 400, 600, 3073, 6000])
def test_staged_row_sums_stay_in_bounds(lib, cols):
    # contiguous rows of 65-512 columns staged in 24 KiB tiles by one bulk
    # copy each, at every 4-byte misalignment of the base
    rows = 3 * (6144 // cols) + 5
    host = inputs.uniform_f32(rows * cols, seed=cols, lo=-1.0, hi=1.0).reshape(rows, cols)
    for offset in range(4):
        x = to_device(host.reshape(-1), offset)
        out = torch.empty(rows, device=DEV)
        assert lib.rdx_rowsum_strided_f32(x.data_ptr(), rows, cols, cols, out.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
        assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)
    assert violations(lib) == 0


@pytest.mark.parametrize("cols", [68, 132, 260, 600, 6000])
def test_rows_staged_stay_in_bounds(lib, cols):
    # rows with a leading dimension, each row bulk-copied into its own slot,
    # at every 4-byte misalignment of the base; the last row ends at the
    # buffer's end
    ld = cols + 3
    rows = 3 * max(1, 6144 // (cols + 32)) + 5
    n = (rows - 1) * ld + cols
    host = inputs.uniform_f32(n, seed=cols, lo=-1.0, hi=1.0)
    full = np.zeros(rows * ld, np.float32)
    full[:n] = host
    ref_rows = full.reshape(rows, ld)[:, :cols]
    for offset in range(4):
        x = to_device(host, offset)
        out = torch.empty(rows, device=DEV)
        assert lib.rdx_rowsum_strided_f32(x.data_ptr(), rows, cols, ld, out.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        tol = 1e-6 * oracle.rowabssum_f32(np.ascontiguousarray(ref_rows)) + 1e-30
        assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(np.ascontiguousarray(ref_rows))) <= tol)
    assert violations(lib) == 0


def test_ladder_stays_in_bounds(lib):
    for v in range(1, 6):
        for n in (1, 255, 257, 513, (1 << 16) + 77):
            host = inputs.normal_f32(n, seed=v)
            x = torch.from_numpy(host).to(DEV)
            nb = lib.rdx_ladder_num_partials(v, n)
            out = torch.empty(nb, device=DEV)
            assert lib.rdx_ladder_partials_f32(v, x.data_ptr(), n, out.data_ptr(), stream()) == 0
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy(), oracle.ladder_partials(v, host))
    assert violations(lib) == 0


def test_ladder_sum_stays_in_bounds(lib):
    for v in range(1, 6):
        for n in (1, 257, 513, (1 << 16) + 77, (1 << 20) + 3):
            host = inputs.normal_f32(n, seed=v + 9)
            x = torch.from_numpy(host).to(DEV)
            nb = lib.rdx_ladder_num_partials(v, n)
            parts = torch.empty(nb, device=DEV)
            out = torch.empty((), device=DEV)
            assert lib.rdx_ladder_sum_f32(v, x.data_ptr(), n, parts.data_ptr(), out.data_ptr(), stream()) == 0
            torch.cuda.synchronize()
            assert np.array_equal(parts.cpu().numpy(), oracle.ladder_partials(v, host))
            check("sum_f32", host, out.item())
    assert violations(lib) == 0


def test_combine_stays_in_bounds(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    for name in ("rdx_combine_f32", "rdx_combine_f32x2", "rdx_combine_i64"):
        getattr(lib, name).argtypes = [vp, i32, vp, vp]
    for p in (1, 2, 257, 4096):
        parts = inputs.normal_f32(2 * p, seed=p)
        x = torch.from_numpy(parts).to(DEV)
        out = torch.empty(2, device=DEV)
        assert lib.rdx_combine_f32(x.data_ptr(), p, out.data_ptr(), stream()) == 0
        assert lib.rdx_combine_f32x2(x.data_ptr(), p, out.data_ptr(), stream()) == 0
        ints = torch.from_numpy(np.arange(p, dtype=np.int64) - 7).to(DEV)
        tot = torch.empty((), dtype=torch.int64, device=DEV)
        assert lib.rdx_combine_i64(ints.data_ptr(), p, tot.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        assert tot.item() == p * (p - 1) // 2 - 7 * p
        assert abs(out[0].item() - oracle.sum_f32(parts[0::2])) <= p * 2.0 ** -24 * oracle.abssum_f32(parts) + 1e-30
    assert violations(lib) == 0
