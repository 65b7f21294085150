"""Reductions split over several GPUs, emulated on one GPU, against the oracle.

The split of reduction_rdx_sum_gb300.shard runs on one GPU: every rank's
chunk through the one-GPU entry point into its slot of a partials array, then
rdx_combine_* in rank order.  That is the set of additions P GPUs make after
their all-gather, so:

* the combine kernels give exactly the rank-order fold that defines them
  (float32 left fold; int64 modulo 2^64), and stay within the recursive-
  summation bound of the float64 oracle;
* a split into P in {1, 2, 3, 8, 72} chunks gives the whole array's sum:
  bit-exact for int32 -> int64, within 1e-6 (float32) / 4e-6 (bfloat16) of the
  summed magnitudes for floats, the same bits on every run, and the bits of
  the one-GPU entry point for P = 1;
* chunks copied into allocations of their own (as each GPU would hold them)
  give the same bits as the emulation's slices of one array;
* row sums split by rows concatenate to the whole matrix's row sums.
"""
import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, build, inputs, shard

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
PARTS = [1, 2, 3, 8, 72]


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    oracle.build()
    torch.cuda.set_device(DEV)
    return abi.load()


def fold_f32(values: np.ndarray) -> np.float32:
    """The rank-order float32 fold ((v0 + v1) + v2) + ... that defines the combine."""
    acc = np.float32(values[0])
    for v in values[1:]:
        acc = np.float32(acc + np.float32(v))
    return acc


@pytest.mark.parametrize("p", [1, 2, 3, 8, 72, 4096])
def test_combine_f32_is_the_rank_order_fold(p):
    parts = inputs.normal_f32(p, seed=p) * np.float32(1000.0)
    got = abi.rdx_combine_f32(torch.from_numpy(parts).to(DEV)).item()
    assert np.float32(got).tobytes() == fold_f32(parts).tobytes()
    bound = (p - 1) * 2.0 ** -24 * oracle.abssum_f32(parts) * 1.01 + 1e-30
    assert abs(got - oracle.sum_f32(parts)) <= bound


@pytest.mark.parametrize("p", [1, 3, 72, 4096])
def test_combine_f32x2_folds_each_component(p):
    pairs = inputs.uniform_f32(2 * p, seed=p, lo=-1.0, hi=1.0).reshape(p, 2)
    got = abi.rdx_combine_f32x2(torch.from_numpy(pairs).to(DEV)).cpu().numpy()
    for c in range(2):
        assert got[c].tobytes() == fold_f32(pairs[:, c]).tobytes()


@pytest.mark.parametrize("p", [1, 2, 72, 4096])
def test_combine_i64_is_exact_modulo_2_64(p):
    rng = np.random.default_rng(p)
    parts = rng.integers(-(2 ** 63), 2 ** 63 - 1, p, dtype=np.int64, endpoint=True)
    got = abi.rdx_combine_i64(torch.from_numpy(parts).to(DEV)).item()
    assert got == oracle.sum_i64(parts)
    wrap = np.array([2 ** 62] * 4 + [5], dtype=np.int64)     # 2^64 + 5 wraps to 5
    assert abi.rdx_combine_i64(torch.from_numpy(wrap).to(DEV)).item() == 5 == oracle.sum_i64(wrap)


def test_combine_rejects_bad_arguments():
    x = torch.zeros(8, dtype=torch.float32, device=DEV)
    with pytest.raises(abi.RdxError):
        abi.rdx_combine_f32(x[:0])
    with pytest.raises(abi.RdxError):
        abi.rdx_combine_f32(torch.zeros(4097, dtype=torch.float32, device=DEV))
    lib = abi.load()
    s = torch.cuda.current_stream(DEV).cuda_stream
    assert lib.rdx_combine_f32(x.data_ptr(), 4, x.data_ptr() + 4, s) == abi.RDX_ERR_INVALID_ARG   # out inside parts
    assert lib.rdx_combine_i64(x.data_ptr() + 4, 1, x.data_ptr() + 16, s) == abi.RDX_ERR_INVALID_ARG  # misaligned


def _host(op: str, n: int) -> np.ndarray:
    if op in ("sum_bf16", "sumsq_bf16", "sum_sumsq_bf16"):
        return inputs.normal_bf16_bits(n, seed=4)
    if op == "sum_i32":
        return inputs.integers_i32(n, seed=2, lo=-(2 ** 31), hi=2 ** 31 - 1)
    return inputs.normal_f32(n, seed=1)


def _device(host: np.ndarray, offset: int) -> torch.Tensor:
    t = torch.from_numpy(host.view(np.int16) if host.dtype == np.uint16 else host)
    buf = torch.empty(host.size + offset, dtype=t.dtype, device=DEV)
    buf[offset:].copy_(t)
    return buf[offset:]


def _check_whole(op: str, host: np.ndarray, got: torch.Tensor):
    v = got.cpu().numpy().astype(np.float64) if op != "sum_i32" else got.item()
    if op == "sum_i32":
        assert v == oracle.sum_i32(host)
        return
    bf = "bf16" in op
    tol = 4e-6 if bf else 1e-6
    s, q = (oracle.sum_bf16, oracle.sumsq_bf16) if bf else (oracle.sum_f32, oracle.sumsq_f32)
    a = oracle.abssum_bf16(host) if bf else oracle.abssum_f32(host)
    if op.startswith("sum_sumsq"):
        assert abs(v[0] - s(host)) <= tol * a + 1e-30
        assert abs(v[1] - q(host)) <= tol * q(host) + 1e-30
    elif op.startswith("sumsq"):
        assert abs(float(v) - q(host)) <= tol * q(host) + 1e-30
    else:
        assert abs(float(v) - s(host)) <= tol * a + 1e-30


SIZES = {"sum_f32": (1 << 22) + 13, "sumsq_f32": (1 << 22) + 13, "sum_i32": (1 << 22) + 5,
         "sum_bf16": (1 << 23) + 7, "sumsq_bf16": (1 << 23) + 7, "sum_sumsq_f32": (1 << 22) + 13,
         "sum_sumsq_bf16": (1 << 23) + 7}


@pytest.mark.parametrize("op", shard.OPS)
@pytest.mark.parametrize("offset", [0, 1])
def test_emulated_split_matches_the_oracle_on_the_whole_array(op, offset):
    host = _host(op, SIZES[op])
    x = _device(host, offset)
    for p in PARTS:
        first = shard.emulate(op, x, p)
        again = shard.emulate(op, x, p)
        torch.cuda.synchronize()
        _check_whole(op, host, first)
        assert first.cpu().numpy().tobytes() == again.cpu().numpy().tobytes(), (op, p)
        if p == 1:
            one = shard.local_partial(op, x)
            assert first.cpu().numpy().tobytes() == one.cpu().numpy().tobytes()


@pytest.mark.parametrize("op", ["sum_f32", "sum_i32", "sum_sumsq_bf16"])
@pytest.mark.parametrize("p", [2, 3, 8])
def test_chunks_in_their_own_allocations_give_the_emulated_bits(op, p):
    """Each GPU holds its chunk in an allocation of its own; with a 16-byte
    aligned array the emulation's slices start 16-byte aligned too, so both
    run the same tiling."""
    host = _host(op, SIZES[op])
    x = _device(host, 0)
    flat = x.reshape(-1)
    dtype, shape = shard.partial_spec(op)
    parts = torch.empty((p, *shape), dtype=dtype, device=DEV)
    for r in range(p):
        own = shard.local_chunk(op, flat, p, r).clone()        # a fresh allocation per rank
        shard.local_partial(op, own, out=parts[r])
    got = shard.combine(op, parts)
    emu = shard.emulate(op, x, p)
    torch.cuda.synchronize()
    assert got.cpu().numpy().tobytes() == emu.cpu().numpy().tobytes()


def test_empty_and_tiny_arrays_split_over_many_ranks():
    for n in (0, 1, 3, 9, 31):
        host = _host("sum_f32", n)
        _check_whole("sum_f32", host, shard.emulate("sum_f32", _device(host, 0), 72))
        z = _host("sum_i32", n)
        assert shard.emulate("sum_i32", _device(z, 0), 72).item() == oracle.sum_i32(z)


@pytest.mark.parametrize("p", [2, 3, 8])
def test_row_sums_split_by_rows(p):
    rows, cols = 1003, 257
    host = inputs.uniform_f32(rows * cols, seed=3, lo=-1.0, hi=1.0).reshape(rows, cols)
    x = torch.from_numpy(host).to(DEV)
    got = torch.cat([shard.sharded_rowsum(shard.local_chunk("rowsum_f32", x, p, r)) for r in range(p)])
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    assert got.numel() == rows
    assert np.all(np.abs(got.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)


@pytest.mark.slow
@pytest.mark.parametrize("op,n", [("sum_sumsq_bf16", (1 << 30) + 7), ("sum_i32", 1 << 28)])
def test_full_size_split_over_eight(op, n):
    host = inputs.normal_bf16_bits(n, seed=4) if "bf16" in op else \
        inputs.integers_i32(n, seed=2, lo=-(1 << 20), hi=1 << 20)
    x = _device(host, 0)
    got = shard.emulate(op, x, 8)
    torch.cuda.synchronize()
    _check_whole(op, host, got)
