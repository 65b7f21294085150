"""Pins of the multi-core CPU baseline (oracle/threads.c): one contiguous chunk
per host thread, each through the single-thread oracle loop, chunk results
added in chunk order.  It is checked against closed forms, against the
single-thread oracle (exactly for integers and row sums, within a float64
bound for the float sums) and for every way of cutting the input."""
import numpy as np
import pytest

import oracle

U64 = 2.0 ** -53

THREADS = [1, 2, 3, 7, 16, 64, 1000]   # 1000 is above the library's 512-thread cap
SIZES = [0, 1, 2, 5, 63, 1000, (1 << 16) + 3]


@pytest.mark.parametrize("threads", THREADS)
@pytest.mark.parametrize("n", SIZES)
def test_closed_forms(n, threads):
    x = np.arange(n, dtype=np.float32)               # exact in float32 and float64
    assert oracle.threaded("sum_f32", x, threads) == n * (n - 1) // 2
    assert oracle.threaded("sumsq_f32", x, threads) == (n - 1) * n * (2 * n - 1) // 6
    i = np.arange(n, dtype=np.int32) - 7
    assert oracle.threaded("sum_i32", i, threads) == n * (n - 1) // 2 - 7 * n
    ones_bf16 = np.full(n, 0x3F80, np.uint16)        # bfloat16 1.0
    assert oracle.threaded("sum_bf16", ones_bf16, threads) == n
    assert oracle.threaded("sumsq_bf16", ones_bf16, threads) == n


@pytest.mark.parametrize("threads", THREADS)
def test_integer_sum_matches_single_thread_exactly(threads):
    x = np.random.default_rng(5).integers(-2**31, 2**31 - 1, size=200_003, endpoint=True, dtype=np.int32)
    assert oracle.threaded("sum_i32", x, threads) == oracle.sum_i32(x) == int(x.astype(np.int64).sum())


@pytest.mark.parametrize("threads", [1, 3, 16])
@pytest.mark.parametrize("op", ["sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16"])
def test_float_sums_within_float64_bound(op, threads):
    rng = np.random.default_rng(6)
    if op.endswith("f32"):
        x = rng.standard_normal(300_007).astype(np.float32)
        scale = oracle.sumsq_f32(x) if op == "sumsq_f32" else oracle.abssum_f32(x)
    else:
        f = rng.standard_normal(300_007).astype(np.float32)
        x = (f.view(np.uint32) >> 16).astype(np.uint16)   # truncated to bfloat16 patterns
        scale = oracle.sumsq_bf16(x) if op == "sumsq_bf16" else oracle.abssum_bf16(x)
    one = getattr(oracle, op)(x)
    many = oracle.threaded(op, x, threads)
    if threads == 1:
        assert many == one                       # the same loop over the same elements
    # each chunk is a Kahan sum (error about 2u of its magnitude); adding the
    # chunk results in float64 adds at most (threads - 1) u of the magnitude
    assert abs(many - one) <= (4 + threads) * U64 * scale


@pytest.mark.parametrize("threads", [1, 2, 5, 16, 1000])
@pytest.mark.parametrize("shape", [(0, 4), (1, 1), (3, 0), (17, 33), (1000, 64)])
def test_rowsum_matches_single_thread_bitwise(shape, threads):
    x = np.random.default_rng(7).uniform(-1, 1, size=shape).astype(np.float32)
    got = oracle.threaded_rowsum_f32(x, threads)
    assert got.shape == (shape[0],)
    assert np.array_equal(got, oracle.rowsum_f32(x))


def test_nonfinite_propagates():
    x = np.ones(1000, np.float32)
    x[999] = np.inf
    assert oracle.threaded("sum_f32", x, 4) == np.inf
    x[0] = -np.inf
    assert np.isnan(oracle.threaded("sum_f32", x, 4))


def test_unknown_op_is_rejected():
    with pytest.raises(KeyError):
        oracle.threaded("max_f32", np.zeros(4, np.float32))
    with pytest.raises(TypeError):
        oracle.threaded("sum_f32", np.zeros(4, np.float64))
