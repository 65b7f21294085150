"""The C-ABI library on the host, without a GPU: it builds for sm_103a, loads,
exports every function include/rdx.h declares, and rejects bad arguments
before making any CUDA call."""
import ctypes
import os

import pytest

from reduction_rdx_sum_gb300 import abi, build

INVALID = abi.RDX_ERR_INVALID_ARG


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def test_exports_every_declared_symbol(lib):
    names = abi.declared_symbols()
    assert {"rdx_sum_f32", "rdx_sum_bf16_f32acc", "rdx_sum_i32_i64", "rdx_rowsum_f32",
            "rdx_sumsq_f32"} <= set(names)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_library_is_in_tree_and_for_sm103a(lib):
    assert os.path.dirname(build.LIB) == os.path.dirname(abi.__file__)
    assert any("arch=compute_103a,code=sm_103a" == f for f in build.NVCC_FLAGS)


def test_status_strings(lib):
    assert abi.status_string(0) == "ok"
    assert abi.status_string(INVALID) == "invalid argument"
    assert "allocation" in abi.status_string(abi.RDX_ERR_ALLOC)
    assert abi.status_string(99) == "unknown status"
    assert lib.rdx_last_cuda_error() == b""


# Argument errors are detected before any CUDA runtime call, so these run
# without a GPU.  A fake device address is fine: nothing dereferences it.
FAKE = 1 << 40


@pytest.mark.parametrize("name,esize,osize", [
    ("rdx_sum_f32", 4, 4), ("rdx_sumsq_f32", 4, 4), ("rdx_sum_bf16_f32acc", 2, 4),
    ("rdx_sumsq_bf16_f32acc", 2, 4), ("rdx_sum_i32_i64", 4, 8), ("rdx_sum_sumsq_f32", 4, 8),
    ("rdx_sum_sumsq_bf16_f32acc", 2, 8), ("rdx_max_f32", 4, 4), ("rdx_max_i32", 4, 4)])
def test_scalar_argument_validation(lib, name, esize, osize):
    fn = getattr(lib, name)
    assert fn(FAKE, -1, FAKE + 4096, None) == INVALID                 # negative n
    assert fn(FAKE, 10, None, None) == INVALID                         # no output
    assert fn(None, 10, FAKE, None) == INVALID                         # no input
    assert fn(FAKE + 1, 10, FAKE + 4096, None) == INVALID              # input not element-aligned
    assert fn(FAKE, 10, FAKE + 4096 + osize // 2, None) == INVALID     # output misaligned
    assert fn(FAKE, 10, FAKE + esize * 3, None) == INVALID             # output inside the input
    assert fn(FAKE, 10, FAKE + esize * 10 - osize, None) == INVALID    # output on the last element
    assert fn(FAKE, 1 << 62, FAKE - 64, None) == INVALID              # size overflow


def test_rowsum_argument_validation(lib):
    f = lib.rdx_rowsum_f32
    assert f(FAKE, -1, 4, FAKE + 4096, None) == INVALID
    assert f(FAKE, 4, -1, FAKE + 4096, None) == INVALID
    assert f(FAKE, 4, 4, None, None) == INVALID
    assert f(None, 4, 4, FAKE, None) == INVALID
    assert f(FAKE + 2, 4, 4, FAKE + 4096, None) == INVALID
    assert f(FAKE, 4, 4, FAKE + 32, None) == INVALID                  # out overlaps x
    assert f(FAKE, 1 << 40, 1 << 40, FAKE - 64, None) == INVALID      # rows*cols overflows
    assert f(None, 0, 5, None, None) == abi.RDX_OK                     # nothing to do


def test_ladder_argument_validation(lib):
    f = lib.rdx_ladder_partials_f32
    assert f(0, FAKE, 10, FAKE + 4096, None) == INVALID
    assert f(6, FAKE, 10, FAKE + 4096, None) == INVALID
    assert f(3, FAKE, -5, FAKE + 4096, None) == INVALID
    assert f(3, None, 10, FAKE, None) == INVALID
    assert f(3, FAKE, 1000, FAKE + 512, None) == INVALID              # partials inside x
    assert f(3, None, 0, None, None) == abi.RDX_OK
    n = lib.rdx_ladder_num_partials
    assert [n(v, 0) for v in range(1, 6)] == [0] * 5
    assert [n(v, 1) for v in range(1, 6)] == [1] * 5
    assert [n(v, 256) for v in range(1, 6)] == [1, 1, 1, 1, 1]
    assert [n(v, 257) for v in range(1, 6)] == [2, 2, 2, 1, 1]
    assert [n(v, 1 << 18) for v in range(1, 6)] == [1024, 1024, 1024, 512, 512]
    assert n(0, 5) == -1 and n(1, -1) == -1


def test_ladder_sum_argument_validation(lib):
    f = lib.rdx_ladder_sum_f32
    part, out = FAKE + 8192, FAKE + 16384
    assert f(0, FAKE, 10, part, out, None) == INVALID                  # bad version
    assert f(6, FAKE, 10, part, out, None) == INVALID
    assert f(3, FAKE, -5, part, out, None) == INVALID                  # negative n
    assert f(3, FAKE, 10, part, None, None) == INVALID                 # no output
    assert f(3, None, 10, part, out, None) == INVALID                  # no input
    assert f(3, FAKE, 10, None, out, None) == INVALID                  # no partials
    assert f(3, FAKE, 10, part, out + 2, None) == INVALID              # output misaligned
    assert f(3, FAKE, 1000, FAKE + 512, out, None) == INVALID          # partials inside x
    assert f(3, FAKE, 1000, part, FAKE + 400, None) == INVALID         # output inside x
    assert f(3, FAKE, 1000, part, part + 4, None) == INVALID           # output inside the partials


def test_python_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(abi, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        abi.load(str(tmp_path / "missing.so"))


def test_workspace_entry_validation(lib):
    f = lib.rdx_reduce_ws
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_size_t, ctypes.c_void_p]
    f.restype = ctypes.c_int
    lib.rdx_workspace_bytes.restype = ctypes.c_size_t
    wsb = lib.rdx_workspace_bytes()
    assert wsb >= 256 + 8192 * 8 and wsb % 256 == 0
    ws = FAKE + (1 << 30)
    assert f(9, FAKE, 10, FAKE + 4096, ws, wsb, None) == INVALID            # bad op
    assert f(-1, FAKE, 10, FAKE + 4096, ws, wsb, None) == INVALID
    assert f(0, FAKE, 10, FAKE + 4096, None, wsb, None) == INVALID          # no workspace
    assert f(0, FAKE, 10, FAKE + 4096, ws, wsb - 1, None) == INVALID        # too small
    assert f(0, FAKE, 10, FAKE + 4096, ws + 16, wsb, None) == INVALID       # not 256-byte aligned
    assert f(0, FAKE, 1 << 20, FAKE + (1 << 23), FAKE + 4096, wsb, None) == INVALID  # workspace inside x
    assert f(0, FAKE, 10, ws + 64, ws, wsb, None) == INVALID                # out inside workspace
    assert f(4, FAKE, 10, FAKE + 4096 + 4, ws, wsb, None) == INVALID        # int64 out misaligned


def test_strided_rowsum_validation(lib):
    f = lib.rdx_rowsum_strided_f32
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(FAKE, 4, 10, 9, FAKE + 4096, None) == INVALID                  # ld < cols
    assert f(FAKE, 4, 10, -1, FAKE + 4096, None) == INVALID
    assert f(FAKE, 4, 10, 20, FAKE + 4 * 65, None) == INVALID               # out inside the last row
    assert f(FAKE, 1 << 40, 8, 1 << 30, FAKE - 64, None) == INVALID         # span overflows
    assert f(None, 0, 10, 20, None, None) == abi.RDX_OK


def test_bank_probe_validation(lib):
    f = lib.rdx_bank_probe
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(-1, 10, FAKE, FAKE + 4096, None) == INVALID
    assert f(10, 10, FAKE, FAKE + 4096, None) == INVALID
    assert f(0, 0, FAKE, FAKE + 4096, None) == INVALID
    assert f(0, (1 << 20) + 1, FAKE, FAKE + 4096, None) == INVALID
    assert f(0, 10, None, FAKE + 4096, None) == INVALID
    assert f(0, 10, FAKE + 4, FAKE + 4096, None) == INVALID          # cycles misaligned
    assert f(0, 10, FAKE, FAKE + 4, None) == INVALID                  # sink overlaps cycles
    lib.rdx_bank_probe_loads_per_iter.restype = ctypes.c_int
    assert lib.rdx_bank_probe_loads_per_iter() >= 1


def test_normal_build_is_unchecked(lib):
    assert lib.rdx_debug_build() == 0
    f = lib.rdx_debug_violations
    f.argtypes, f.restype = [ctypes.c_void_p, ctypes.c_int], ctypes.c_int
    count = ctypes.c_uint64(7)
    assert f(ctypes.byref(count), 0) == abi.RDX_OK and count.value == 0   # no CUDA call in a normal build
    assert f(None, 0) == INVALID


def test_kernel_counts_per_call(lib):
    # tiles of 64 KiB and more finish in a second kernel; shorter ones in the last block
    assert abi.rdx_reduce_kernels("sum_f32", 0) == 1
    assert abi.rdx_reduce_kernels("sum_f32", 1 << 20) == 1
    assert abi.rdx_reduce_kernels("sum_f32", (1 << 22) + 13) == 1
    assert abi.rdx_reduce_kernels("sum_f32", (1 << 24) + 13) == 2
    assert abi.rdx_reduce_kernels("sum_i32", 1 << 28) == 2
    assert abi.rdx_reduce_kernels("sum_bf16", (1 << 30) + 7) == 2
    assert abi.rdx_reduce_kernels("max_i32", 1 << 28) == 2
    assert abi.rdx_reduce_kernels(99, 10) == -1 and abi.rdx_reduce_kernels("sum_f32", -1) == -1
    assert abi.rdx_rowsum_kernels(0, 5) == 0
    assert abi.rdx_rowsum_kernels(8192, 32768) == 1 and abi.rdx_rowsum_kernels(1 << 20, 256) == 1
    assert abi.rdx_rowsum_kernels(4, 1 << 26) == 2
    assert abi.rdx_rowsum_kernels(-1, 5) == -1


def test_stage_timeout_entry_validation(lib):
    # every argument check comes before any CUDA call
    assert lib.rdx_wait_timeouts(None, 0) == INVALID
    f = lib.rdx_debug_stage_timeout
    assert f(None, 100, 16, FAKE + 65536, None) == INVALID
    assert f(FAKE, 100, 16, None, None) == INVALID
    assert f(FAKE, 100, 0, FAKE + 65536, None) == INVALID              # cols outside 1..63
    assert f(FAKE, 100, 64, FAKE + 65536, None) == INVALID
    assert f(FAKE, 0, 16, FAKE + 65536, None) == INVALID               # no rows
    assert f(FAKE, 385, 16, FAKE + 65536, None) == INVALID             # more than one 6144-float tile
    assert f(FAKE, 1 << 62, 16, FAKE + 65536, None) == INVALID         # rows far beyond, no overflow
    assert f(FAKE, 1, 3, FAKE + 65536, None) == INVALID                # fewer than 4 floats
    assert f(FAKE + 4, 100, 16, FAKE + 65536, None) == INVALID         # x not 16-byte aligned
    assert f(FAKE, 100, 16, FAKE + 65538, None) == INVALID             # out misaligned
    assert f(FAKE, 100, 16, FAKE + 64, None) == INVALID                # out inside x
