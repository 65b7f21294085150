"""Seeded random shapes against the oracle: row sums over every kernel
choice (narrow plain and rotated, short rows, a warp per row, a block per
row, split rows; contiguous and with a leading dimension; every 4-byte base
offset), and scalar reductions over sizes and offsets around every tiling
threshold.  Each case is small; the seeds make every run the same."""
import math

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, inputs

from test_parity_gpu import DEV, VEC, check, host_input, to_device

pytestmark = pytest.mark.gpu

MAX_ELEMS = 1 << 22  # per case


def _row_shape(rng):
    cols = int(math.exp(rng.uniform(0.0, math.log(40000.0))))
    cols = max(cols, 1)
    rows = int(math.exp(rng.uniform(0.0, math.log(5000.0))))
    rows = max(1, min(rows, MAX_ELEMS // (cols + 17)))
    ld = cols if rng.random() < 0.6 else cols + int(rng.integers(1, 18))
    offset = int(rng.integers(0, 4))
    return rows, cols, ld, offset


@pytest.mark.parametrize("case", range(120))
def test_random_row_shapes(case):
    rng = np.random.default_rng(1000 + case)
    rows, cols, ld, offset = _row_shape(rng)
    exact = case % 3 == 0
    if exact:   # small integers: every row sum exact in float32
        full = (rng.integers(-7, 8, size=rows * ld)).astype(np.float32)
    else:
        full = inputs.uniform_f32(rows * ld, seed=case, lo=-1.0, hi=1.0)
    buf = torch.empty(rows * ld + offset, dtype=torch.float32, device=DEV)
    buf[offset:].copy_(torch.from_numpy(full))
    x = buf[offset:].view(rows, ld)[:, :cols]
    got = (abi.rdx_rowsum_f32(x) if ld == cols else abi.rdx_rowsum_strided_f32(x)).cpu().numpy()
    host = np.ascontiguousarray(full.reshape(rows, ld)[:, :cols])
    if exact:
        assert np.array_equal(got.astype(np.int64), host.astype(np.int64).sum(axis=1)), (rows, cols, ld, offset)
    else:
        ref = oracle.rowsum_f32(host)
        tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
        bad = np.nonzero(~(np.abs(got.astype(np.float64) - ref) <= tol))[0]
        assert bad.size == 0, (rows, cols, ld, offset, bad[:5])


OPS = ["sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16", "sum_i32"]


@pytest.mark.parametrize("case", range(120))
def test_random_scalar_sizes(case):
    rng = np.random.default_rng(5000 + case)
    op = OPS[case % len(OPS)]
    n = int(math.exp(rng.uniform(0.0, math.log(float(1 << 24)))))
    offset = int(rng.integers(0, VEC[op]))
    host = host_input(op, n, seed=case)
    x = to_device(host, offset)
    got = abi.SCALAR_OPS[op](x).item()
    check(op, host, got)
    assert abi.SCALAR_OPS[op](x).item() == got  # the same bits again


@pytest.mark.parametrize("case", range(40))
def test_random_maxima(case):
    rng = np.random.default_rng(9000 + case)
    n = int(math.exp(rng.uniform(0.0, math.log(float(1 << 23)))))
    offset = int(rng.integers(0, 4))
    f = inputs.normal_f32(n, seed=case) * np.float32(rng.choice([1e-40, 1.0, 1e30]))
    z = inputs.integers_i32(n, seed=case, lo=-(2 ** 31), hi=2 ** 31 - 1)
    assert abi.rdx_max_f32(to_device(f, offset)).item() == oracle.max_f32(f)
    assert abi.rdx_max_i32(to_device(z, offset)).item() == oracle.max_i32(z)


@pytest.mark.parametrize("case", range(24))
def test_random_large_scalar_sizes(case):
    """Sizes of 64-256 MiB, where the tiles' partials are added by the
    separate finish kernel (tiles of 64 KiB and more)."""
    rng = np.random.default_rng(7000 + case)
    op = OPS[case % len(OPS)]
    lo_n = (1 << 24) * (2 if "bf16" in op else 1)
    n = int(math.exp(rng.uniform(math.log(float(lo_n)), math.log(float(1 << 26)))))
    offset = int(rng.integers(0, VEC[op]))
    host = host_input(op, n, seed=case)
    x = to_device(host, offset)
    assert abi.rdx_reduce_kernels(op, n) == 2
    got = abi.SCALAR_OPS[op](x).item()
    check(op, host, got)
    assert abi.SCALAR_OPS[op](x).item() == got  # the same bits again


@pytest.mark.parametrize("case", range(40))
def test_random_splits(case):
    """The sum split into a random number of chunks (as over that many GPUs),
    emulated on this GPU, against the oracle on the whole array."""
    from reduction_rdx_sum_gb300 import shard

    rng = np.random.default_rng(11000 + case)
    op = OPS[case % len(OPS)]
    n = int(math.exp(rng.uniform(0.0, math.log(float(1 << 23)))))
    parts = int(rng.integers(1, 81))
    offset = int(rng.integers(0, VEC[op]))
    host = host_input(op, n, seed=case)
    got = shard.emulate(op, to_device(host, offset), parts).item()
    check(op, host, got)


@pytest.mark.parametrize("case", range(40))
def test_random_pairs(case):
    """The one-pass [sum, sum of squares] pairs over random sizes, offsets and
    scales.  At scale 1e20 every square passes the float32 range, so the sum
    of squares is +Inf (the correctly rounded float32 result) while the sum
    stays finite; at 1e-30 the squares underflow to zero or subnormals."""
    rng = np.random.default_rng(13000 + case)
    n = max(1, int(math.exp(rng.uniform(0.0, math.log(float(1 << 23))))))
    offset = int(rng.integers(0, 4))
    scale = np.float32(rng.choice([1e-30, 1.0, 1e20]))
    f = inputs.normal_f32(n, seed=case) * scale
    s, q = abi.rdx_sum_sumsq_f32(to_device(f, offset)).cpu().numpy().astype(np.float64)
    assert abs(s - oracle.sum_f32(f)) <= 1e-6 * oracle.abssum_f32(f) + 1e-30
    if scale == np.float32(1e20):
        assert q == math.inf
    else:
        ref = oracle.sumsq_f32(f)
        assert abs(q - ref) <= 1e-6 * ref + 1e-30
    b = inputs.normal_bf16_bits(n, seed=case)
    s, q = abi.rdx_sum_sumsq_bf16_f32acc(to_device(b, int(rng.integers(0, 8)))).cpu().numpy().astype(np.float64)
    assert abs(s - oracle.sum_bf16(b)) <= 4e-6 * oracle.abssum_bf16(b) + 1e-30
    ref = oracle.sumsq_bf16(b)
    assert abs(q - ref) <= 4e-6 * ref + 1e-30
