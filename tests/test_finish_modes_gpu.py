"""The two finishes of the tiled reductions give the same bits.

Inputs cut into long tiles (64 KiB and more: 64 MiB and up) finish in a
kernel of their own, launched behind the tiles' grid; shorter tiles finish in
the grid's last block.  Both run the same fixed-order pass over the same
partials, so a library built with the separate finish switched off
(-DRDX_SEPARATE_FINISH_MIN_TILE set past any tile) must return the same bits
as the normal one, for every op, at aligned and misaligned bases, and for the
row sums of few long rows.  Both are also checked against the oracle.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, build, inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ONE_KERNEL = os.path.join(os.path.dirname(build.LIB), "..", "_build", "librdx_onekernel.so")
OUT = {"sum_i32": torch.int64, "max_i32": torch.int32}


@pytest.fixture(scope="module")
def libs():
    path = build.build(defines=["-DRDX_SEPARATE_FINISH_MIN_TILE=4611686018427387904"],
                       out=os.path.abspath(ONE_KERNEL))
    oracle.build()
    torch.cuda.set_device(DEV)
    one = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    one.rdx_reduce_ws.argtypes = [i32, vp, i64, vp, vp, ctypes.c_size_t, vp]
    one.rdx_workspace_bytes.restype = ctypes.c_size_t
    one.rdx_rowsum_f32.argtypes = [vp, i64, i64, vp, vp]
    return abi.load(), one


def _host(op, n):
    if "bf16" in op:
        return inputs.normal_bf16_bits(n, seed=4)
    if op.endswith("i32"):
        return inputs.integers_i32(n, seed=2, lo=-(2 ** 31), hi=2 ** 31 - 1)
    return inputs.normal_f32(n, seed=1)


def _device(host, offset):
    t = torch.from_numpy(host.view(np.int16) if host.dtype == np.uint16 else host)
    buf = torch.empty(host.size + offset, dtype=t.dtype, device=DEV)
    buf[offset:].copy_(t)
    return buf[offset:]


OPS = ["sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16", "sum_i32", "sum_sumsq_f32", "sum_sumsq_bf16",
       "max_f32", "max_i32"]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [(1 << 24) + 13, (1 << 26) + 3])
def test_separate_and_last_block_finish_agree_bitwise(libs, op, n):
    lib, one = libs
    host = _host(op, n)
    s = torch.cuda.current_stream(DEV).cuda_stream
    shape = (2,) if op.startswith("sum_sumsq") else ()
    dt = OUT.get(op, torch.float32)
    ws_a = torch.zeros(lib.rdx_workspace_bytes(), dtype=torch.uint8, device=DEV)
    ws_b = torch.zeros(one.rdx_workspace_bytes(), dtype=torch.uint8, device=DEV)
    for offset in (0, 1):
        x = _device(host, offset)
        a = torch.full(shape, -1, dtype=dt, device=DEV)
        b = torch.full(shape, -1, dtype=dt, device=DEV)
        code = abi.OP_CODES[op]
        assert lib.rdx_reduce_ws(code, x.data_ptr(), n, a.data_ptr(), ws_a.data_ptr(), ws_a.numel(), s) == 0
        assert one.rdx_reduce_ws(code, x.data_ptr(), n, b.data_ptr(), ws_b.data_ptr(), ws_b.numel(), s) == 0
        named = abi.SCALAR_OPS[op](x) if op in abi.SCALAR_OPS else abi.PAIR_OPS[op.split("_")[-1]](x)
        torch.cuda.synchronize()
        assert a.cpu().numpy().tobytes() == b.cpu().numpy().tobytes(), (op, n, offset)
        assert named.cpu().numpy().tobytes() == a.cpu().numpy().tobytes()
        v = a.cpu().numpy()
        if op == "sum_i32":
            assert int(v) == oracle.sum_i32(host)
        elif op == "max_i32":
            assert int(v) == oracle.max_i32(host)
        elif op == "max_f32":
            assert float(v) == oracle.max_f32(host)
        else:
            bf = "bf16" in op
            tol = 4e-6 if bf else 1e-6
            s_ref = oracle.sum_bf16(host) if bf else oracle.sum_f32(host)
            q_ref = oracle.sumsq_bf16(host) if bf else oracle.sumsq_f32(host)
            a_ref = oracle.abssum_bf16(host) if bf else oracle.abssum_f32(host)
            if op.startswith("sum_sumsq"):
                assert abs(float(v[0]) - s_ref) <= tol * a_ref + 1e-30
                assert abs(float(v[1]) - q_ref) <= tol * q_ref + 1e-30
            elif op.startswith("sumsq"):
                assert abs(float(v) - q_ref) <= tol * q_ref + 1e-30
            else:
                assert abs(float(v) - s_ref) <= tol * a_ref + 1e-30


@pytest.mark.parametrize("shape", [(4, 1 << 24), (3, (1 << 24) + 5)], ids=str)
def test_split_rows_agree_bitwise(libs, shape):
    lib, one = libs
    rows, cols = shape
    host = inputs.uniform_f32(rows * cols, seed=3, lo=-1.0, hi=1.0).reshape(rows, cols)
    x = torch.from_numpy(host).to(DEV)
    s = torch.cuda.current_stream(DEV).cuda_stream
    a = torch.empty(rows, device=DEV)
    b = torch.empty(rows, device=DEV)
    assert lib.rdx_rowsum_f32(x.data_ptr(), rows, cols, a.data_ptr(), s) == 0
    assert one.rdx_rowsum_f32(x.data_ptr(), rows, cols, b.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert a.cpu().numpy().tobytes() == b.cpu().numpy().tobytes()
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    assert np.all(np.abs(a.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)
