"""Host side of the reductions split over several GPUs, on the CPU.

* rdx_shard_range (the C library's host-only chunking rule) tiles [0, n) with
  contiguous, balanced chunks whose starts are whole granules, for sizes
  around every vector boundary and rank counts up to a 72-GPU domain.
* Two and three gloo ranks run the exchange of reduction_rdx_sum_gb300.shard:
  each rank takes its chunk of a seeded array, computes the chunk's partial
  with the oracle (standing in for the GPU entry point, which needs a GPU),
  and gather_partials returns every rank's partial in rank order, the same
  on every rank.  The sum of the gathered partials is the whole array's sum:
  exactly for int32 -> int64, within the float32 tolerance for float32, and
  row sums split by rows concatenate to the whole matrix's row sums.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from reduction_rdx_sum_gb300 import abi, build  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def _sizes():
    out = {0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 63, 64, 65, 127, 1000, 4093, 4096, 4099,
           (1 << 24) + 13, (1 << 30) + 7}
    for g in (4, 8):
        for k in (1, 2, 3, 71, 72, 73, 1024):
            out.update({k * g - 1, k * g, k * g + 1})
    return sorted(out)


@pytest.mark.parametrize("granule", [1, 4, 8])
@pytest.mark.parametrize("parts", [1, 2, 3, 7, 8, 72])
def test_chunks_tile_the_range(lib, parts, granule):
    for n in _sizes():
        chunks = [abi.rdx_shard_range(n, parts, r, granule) for r in range(parts)]
        assert chunks[0][0] == 0 and chunks[-1][1] == n
        for (lo, hi), (lo2, _) in zip(chunks, chunks[1:]):
            assert lo <= hi == lo2
        for r, (lo, hi) in enumerate(chunks):
            assert lo % granule == 0
            if r < parts - 1:
                assert hi % granule == 0
        # balanced: whole granules per rank differ by at most one, more on lower ranks
        g = [(hi - lo) // granule for lo, hi in chunks[:-1]] + [(chunks[-1][1] - chunks[-1][0]) // granule]
        assert max(g) - min(g) <= 1 and g == sorted(g, reverse=True)
        assert sum(g) == n // granule
        assert chunks[-1][1] - chunks[-1][0] - g[-1] * granule == n % granule


def test_shard_range_rejects_bad_arguments(lib):
    for args in ((-1, 2, 0, 4), (10, 0, 0, 4), (10, 2, 2, 4), (10, 2, -1, 4), (10, 2, 0, 0)):
        with pytest.raises(abi.RdxError):
            abi.rdx_shard_range(*args)


def test_combine_limit_is_exported(lib):
    assert abi.rdx_combine_max_parts() == 4096


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from reduction_rdx_sum_gb300 import inputs, shard

    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = {}
    # int32 -> int64: the chunk's exact partial
    z = inputs.integers_i32(100_003, seed=2, lo=-(2 ** 31), hi=2 ** 31 - 1)
    lo, hi = shard.shard_range("sum_i32", z.size, world, rank)
    got = shard.gather_partials(torch.tensor(oracle.sum_i32(z[lo:hi]), dtype=torch.int64))
    out["i64"] = got.tolist()
    out["i64_rank_order"] = shard.gather_partials(torch.tensor(rank, dtype=torch.int64)).tolist()
    # float32: the chunk's partial rounded to float32, as the GPU returns it
    x = inputs.normal_f32(200_013, seed=1)
    lo, hi = shard.shard_range("sum_f32", x.size, world, rank)
    out["f32"] = shard.gather_partials(torch.tensor(oracle.sum_f32(x[lo:hi]), dtype=torch.float32)).tolist()
    # [sum, sum of squares] pairs of bfloat16 input
    b = inputs.normal_bf16_bits(50_007, seed=4)
    lo, hi = shard.shard_range("sum_sumsq_bf16", b.size, world, rank)
    pair = torch.tensor([oracle.sum_bf16(b[lo:hi]), oracle.sumsq_bf16(b[lo:hi])], dtype=torch.float32)
    out["f32x2"] = shard.gather_partials(pair).tolist()
    # rows: the rank's slice of the row sums, no exchange needed
    m = inputs.uniform_f32(37 * 129, seed=3, lo=-1.0, hi=1.0).reshape(37, 129)
    rows = shard.local_chunk("rowsum_f32", torch.from_numpy(m), world, rank).numpy()
    out["rows"] = oracle.rowsum_f32(rows).tolist()
    results[rank] = out
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_with_gloo_ranks(lib, world):
    import oracle
    from reduction_rdx_sum_gb300 import inputs

    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(results)
    # every rank holds the same gathered partials, in rank order
    for key in ("i64", "i64_rank_order", "f32", "f32x2"):
        assert all(res[r][key] == res[0][key] for r in range(world)), key
    assert res[0]["i64_rank_order"] == list(range(world))
    assert len(res[0]["i64"]) == world

    z = inputs.integers_i32(100_003, seed=2, lo=-(2 ** 31), hi=2 ** 31 - 1)
    assert oracle.sum_i64(np.array(res[0]["i64"], dtype=np.int64)) == oracle.sum_i32(z)
    x = inputs.normal_f32(200_013, seed=1)
    parts = np.array(res[0]["f32"], dtype=np.float32)
    assert abs(oracle.sum_f32(parts) - oracle.sum_f32(x)) <= 1e-6 * oracle.abssum_f32(x)
    b = inputs.normal_bf16_bits(50_007, seed=4)
    pairs = np.array(res[0]["f32x2"], dtype=np.float32)
    assert abs(oracle.sum_f32(pairs[:, 0]) - oracle.sum_bf16(b)) <= 4e-6 * oracle.abssum_bf16(b)
    q = oracle.sumsq_bf16(b)
    assert abs(oracle.sum_f32(pairs[:, 1]) - q) <= 4e-6 * q
    m = inputs.uniform_f32(37 * 129, seed=3, lo=-1.0, hi=1.0).reshape(37, 129)
    rows = np.concatenate([np.array(res[r]["rows"]) for r in range(world)])
    assert np.array_equal(rows, oracle.rowsum_f32(m))


def test_chunks_tile_the_range_for_random_arguments(lib):
    """Property check over random (n, parts, granule): contiguous chunks that
    tile [0, n), whole granules except the last chunk's tail, balanced."""
    hypothesis = pytest.importorskip("hypothesis")
    st = hypothesis.strategies

    @hypothesis.settings(max_examples=200, deadline=None)
    @hypothesis.given(n=st.integers(0, 1 << 40), parts=st.integers(1, 1024), granule=st.sampled_from([1, 2, 4, 8, 16]))
    def check(n, parts, granule):
        chunks = [abi.rdx_shard_range(n, parts, r, granule) for r in range(parts)]
        assert chunks[0][0] == 0 and chunks[-1][1] == n
        assert all(hi == lo2 for (_, hi), (lo2, _) in zip(chunks, chunks[1:]))
        assert all(lo % granule == 0 and lo <= hi for lo, hi in chunks)
        assert all(hi % granule == 0 for _, hi in chunks[:-1])
        counts = [(hi - lo) // granule for lo, hi in chunks]
        assert max(counts) - min(counts) <= 1 and counts == sorted(counts, reverse=True)

    check()
