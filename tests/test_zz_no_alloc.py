"""rdx_sum_f32_noalloc: the float32 sum that allocates no device memory (for
callers inside a framework that owns all device memory, latency-critical
callers, and fixed-budget programs).  Checked against rdx_sum_f32, through the
C ABI, on two calls in a row that share the library's static scratch.

This file is collected last on purpose: it must pass both alone in a fresh
process (the first call on the device does the one-time set-up) and after
every other test has run.
"""
import ctypes

import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, build, inputs

pytestmark = pytest.mark.gpu


def test_noalloc_sum_matches_rdx_sum_f32_on_two_calls_in_a_row():
    build.build()
    oracle.build()
    lib = abi.load()
    noalloc = lib.rdx_sum_f32_noalloc
    noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    noalloc.restype = ctypes.c_int
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream

    # two inputs of different sizes: the second call reuses the scratch the
    # first one left behind
    hosts = [inputs.normal_f32((1 << 24) + 13, seed=1), inputs.uniform_f32(1_000_003, seed=5, lo=-1.0, hi=1.0)]
    xs = [torch.from_numpy(h).to(dev) for h in hosts]
    refs = [torch.empty((), dtype=torch.float32, device=dev) for _ in xs]
    gots = [torch.full((), float("nan"), dtype=torch.float32, device=dev) for _ in xs]
    for x, ref in zip(xs, refs):
        assert lib.rdx_sum_f32(x.data_ptr(), x.numel(), ref.data_ptr(), stream) == 0
    torch.cuda.synchronize()
    for x, got in zip(xs, gots):           # the two no-allocation calls, back to back
        assert noalloc(x.data_ptr(), x.numel(), got.data_ptr(), stream) == 0, lib.rdx_last_cuda_error()
    torch.cuda.synchronize()
    for h, ref, got in zip(hosts, refs, gots):
        tol = 1e-6 * oracle.abssum_f32(h) + 1e-30
        assert abs(got.item() - ref.item()) <= tol, (got.item(), ref.item(), tol)
