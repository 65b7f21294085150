"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: integer sums bit-exact; float32 input |gpu - oracle| <= 1e-6 * sum|x_i|
+ 1e-30; bfloat16 input 4e-6 * sum|x_i|; sums of squares the same factors
times sum x_i^2; row sums per row against that row's sum |x|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
FACTOR = {"sum_f32": 1e-6, "sumsq_f32": 1e-6, "sum_bf16": 4e-6, "sumsq_bf16": 4e-6}
OPS = ["sum_f32", "sumsq_f32", "sum_bf16", "sumsq_bf16", "sum_i32"]
VEC = {"sum_f32": 4, "sumsq_f32": 4, "sum_bf16": 8, "sumsq_bf16": 8, "sum_i32": 4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from reduction_rdx_sum_gb300 import build

    build.build()
    oracle.build()
    abi.load()
    torch.cuda.set_device(DEV)


def host_input(op, n, seed):
    if op in ("sum_f32", "sumsq_f32"):
        return inputs.normal_f32(n, seed)
    if op in ("sum_bf16", "sumsq_bf16"):
        return inputs.normal_bf16_bits(n, seed)
    return inputs.integers_i32(n, seed, -(2 ** 31), 2 ** 31 - 1)  # full range: int64 carries


def to_device(host, offset=0):
    """Device copy of host; with offset > 0 the returned view starts offset
    elements into an allocation (its address is misaligned by that much)."""
    a = host.view(np.int16) if host.dtype == np.uint16 else host
    buf = torch.empty(a.size + offset, dtype=torch.from_numpy(a[:0]).dtype, device=DEV)
    view = buf[offset:]
    view.copy_(torch.from_numpy(a))
    return view


def reference(op, host):
    """(oracle value, tolerance) for a scalar op."""
    if op == "sum_i32":
        return oracle.sum_i32(host), 0
    if op == "sum_f32":
        return oracle.sum_f32(host), FACTOR[op] * oracle.abssum_f32(host) + 1e-30
    if op == "sumsq_f32":
        v = oracle.sumsq_f32(host)
        return v, FACTOR[op] * v + 1e-30
    if op == "sum_bf16":
        return oracle.sum_bf16(host), FACTOR[op] * oracle.abssum_bf16(host) + 1e-30
    v = oracle.sumsq_bf16(host)
    return v, FACTOR[op] * v + 1e-30


def check(op, host, got):
    ref, tol = reference(op, host)
    if op == "sum_i32":
        assert int(got) == ref
    else:
        assert abs(float(got) - ref) <= tol, (float(got), ref, tol)


SIZES = [0, 1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511,
         512, 513, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4096, 4097, 8191, 8193, 65535, 65536, 65537,
         262143, 262144, 262145, (1 << 20) - 1, 1 << 20, (1 << 20) + 1, 1_000_003, (1 << 22) + 13,
         (1 << 24) + 13]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", SIZES)
def test_scalar_parity(op, n):
    host = host_input(op, n, seed=n % 97)
    got = abi.SCALAR_OPS[op](to_device(host)).item()
    check(op, host, got)


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [1, 3, 5, 9, 100, 4097, (1 << 20) + 3])
def test_scalar_parity_misaligned_base(op, n):
    host = host_input(op, n, seed=7)
    for offset in range(1, VEC[op]):
        got = abi.SCALAR_OPS[op](to_device(host, offset)).item()
        check(op, host, got)


# Inputs of 4096 tiles or more (about 256 MiB) take the deeper kernel variant
# (8 loads in flight per thread, 4 blocks per SM).  4095 * 4096 whole 16-byte
# vectors is the last size on the shallow side; one more vector crosses over.
EDGE_VECTORS = 4095 * 4096


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("extra", [0, 1, 3])
def test_scalar_parity_across_the_deep_variant_threshold(op, extra):
    per_vec = VEC[op]
    n = EDGE_VECTORS * per_vec + extra * per_vec + (extra % 2) * (per_vec - 1)  # ragged tail when extra is odd
    host = host_input(op, n, seed=extra + 11)
    for offset in (0, 1):
        x = to_device(host, offset)
        a = abi.SCALAR_OPS[op](x).item()
        check(op, host, a)
        assert abi.SCALAR_OPS[op](x).item() == a  # bitwise reproducible


def test_empty_input_writes_zero():
    for op in OPS:
        dt = {"sum_f32": torch.float32, "sumsq_f32": torch.float32, "sum_bf16": torch.bfloat16,
              "sumsq_bf16": torch.bfloat16, "sum_i32": torch.int32}[op]
        out = torch.full((), 123, dtype=torch.int64 if op == "sum_i32" else torch.float32, device=DEV)
        abi.SCALAR_OPS[op](torch.empty(0, dtype=dt, device=DEV), out=out)
        assert out.item() == 0


def test_page_worked_example_sum():
    # "03_shared_memory_sync_reduction.py", demo 3: in[i] = i mod 7, exact sums
    for n, total in ((1 << 14, 49146), (1 << 18, 786429)):
        x = torch.from_numpy((np.arange(n) % 7).astype(np.float32)).to(DEV)
        assert abi.rdx_sum_f32(x).item() == total


def test_integer_extremes_exact():
    n = (1 << 24) + 5
    for v in (2 ** 31 - 1, -(2 ** 31)):
        x = torch.full((n,), v, dtype=torch.int32, device=DEV)
        assert abi.rdx_sum_i32_i64(x).item() == v * n


def test_integer_accumulator_word_left_clear_between_ops():
    # The int64 sum and the int32 maximum finish through one accumulator word
    # of the stream's workspace; every call must leave it clear for the next,
    # whichever op comes next.  All -2^31 is the maximum whose word key is 0.
    hosts = [inputs.integers_i32((1 << 22) + k, seed=40 + k, lo=-(2 ** 31), hi=2 ** 31 - 1) for k in range(3)]
    xs = [to_device(h, offset=k) for k, h in enumerate(hosts)]
    low = torch.full(((1 << 20) + 3,), -(2 ** 31), dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    for rep in range(3):
        for h, x in zip(hosts, xs):
            assert abi.rdx_sum_i32_i64(x).item() == oracle.sum_i32(h)
            assert abi.rdx_max_i32(x).item() == oracle.max_i32(h)
        assert abi.rdx_max_i32(low).item() == -(2 ** 31)
        assert abi.rdx_sum_i32_i64(low).item() == -(2 ** 31) * low.numel()
        with torch.cuda.stream(side):
            got = abi.rdx_max_i32(xs[rep], stream=side)
        side.synchronize()
        assert got.item() == oracle.max_i32(hosts[rep])


def test_subnormal_inputs_are_not_flushed():
    # n copies of the smallest subnormal: every partial sum is a multiple of
    # it well inside float32's exact range, so the sum is exactly n times it
    # in any order (a build that flushed subnormals to zero would return 0)
    n = (1 << 20) + 3
    tiny = np.float32(2.0 ** -149)                      # smallest float32 subnormal
    x = np.full(n, tiny, np.float32)
    assert abi.rdx_sum_f32(to_device(x, 1)).item() == n * 2.0 ** -149 == oracle.sum_f32(x)
    rows = x[: 1000 * 1000].reshape(1000, 1000)
    assert np.all(abi.rdx_rowsum_f32(to_device(rows.reshape(-1)).view(1000, 1000)).cpu().numpy() == np.float32(1000 * 2.0 ** -149))
    b = np.full(n, 0x0001, np.uint16)                    # smallest bfloat16 subnormal, 2^-133
    assert abi.rdx_sum_bf16_f32acc(to_device(b, 3)).item() == n * 2.0 ** -133 == oracle.sum_bf16(b)
    assert abi.rdx_max_f32(to_device(x)).item() == 2.0 ** -149


def test_overflow_gives_infinity():
    # same-sign terms whose exact sum passes the largest float32: the float32
    # result, correctly rounded, is the infinity of their sign, whatever the
    # order of the additions
    n = (1 << 20) + 1
    x = np.full(n, np.float32(1e33), np.float32)        # exact sum 1.05e39 > 3.4e38
    assert abi.rdx_sum_f32(to_device(x)).item() == math.inf
    assert abi.rdx_sum_f32(to_device(-x)).item() == -math.inf
    assert abi.rdx_sumsq_f32(to_device(np.full(n, np.float32(1e17), np.float32))).item() == math.inf
    # the one-pass pair: the sum stays finite while the sum of squares overflows
    y = inputs.normal_f32(n, seed=9) * np.float32(1e20)  # sum of squares about 1e46
    pair = abi.rdx_sum_sumsq_f32(to_device(y, 1)).cpu().numpy().astype(np.float64)
    assert abs(pair[0] - oracle.sum_f32(y)) <= 1e-6 * oracle.abssum_f32(y) and pair[1] == math.inf
    yb = np.full(n, 0x5F80, np.uint16)                    # bfloat16 2^64: squares 2^128 pass the float32 range
    pair = abi.rdx_sum_sumsq_bf16_f32acc(to_device(yb, 3)).cpu().numpy().astype(np.float64)
    assert pair[0] == n * 2.0 ** 64 and pair[1] == math.inf
    rows = np.full(4 * 65536, np.float32(1e34), np.float32)  # each row's exact sum 6.6e38
    assert abi.rdx_rowsum_f32(to_device(rows).view(4, 65536)).tolist() == [math.inf] * 4


def test_nonfinite_propagation():
    n = 100_003
    for pos in (0, 5, n // 2, n - 1):
        x = torch.ones(n, dtype=torch.float32, device=DEV)
        x[pos] = math.inf
        assert abi.rdx_sum_f32(x).item() == math.inf
        assert abi.rdx_sumsq_f32(x).item() == math.inf
        x[(pos + 7) % n] = -math.inf
        assert math.isnan(abi.rdx_sum_f32(x).item())
        x = torch.ones(n, dtype=torch.float32, device=DEV)
        x[pos] = math.nan
        assert math.isnan(abi.rdx_sum_f32(x).item())
        b = torch.ones(n, dtype=torch.bfloat16, device=DEV)
        b[pos] = -math.inf
        assert abi.rdx_sum_bf16_f32acc(b).item() == -math.inf


# ---------------------------------------------------------------------------
# one-pass sum and sum of squares
# ---------------------------------------------------------------------------

def check_pair(kind, host, got):
    s_op, q_op = ("sum_f32", "sumsq_f32") if kind == "f32" else ("sum_bf16", "sumsq_bf16")
    check(s_op, host, got[0])
    check(q_op, host, got[1])


@pytest.mark.parametrize("kind", ["f32", "bf16"])
@pytest.mark.parametrize("n", SIZES)
def test_sum_sumsq_parity(kind, n):
    host = host_input("sum_f32" if kind == "f32" else "sum_bf16", n, seed=n % 89)
    got = abi.PAIR_OPS[kind](to_device(host)).tolist()
    check_pair(kind, host, got)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_sum_sumsq_misaligned_and_deterministic(kind):
    op = "sum_f32" if kind == "f32" else "sum_bf16"
    for n in (5, 4097, (1 << 20) + 3):
        host = host_input(op, n, seed=3)
        for offset in range(1, VEC[op]):
            check_pair(kind, host, abi.PAIR_OPS[kind](to_device(host, offset)).tolist())
    x = to_device(host_input(op, (1 << 24) + 13, seed=1))
    first = abi.PAIR_OPS[kind](x)
    for _ in range(5):
        assert torch.equal(abi.PAIR_OPS[kind](x).view(torch.int32), first.view(torch.int32))


@pytest.mark.slow
@pytest.mark.parametrize("w", (inputs.CFG2_SUM_F32, inputs.CFG5_SUM_BF16), ids=lambda w: w.name)
def test_config_sum_sumsq(w):
    host = workload(w)
    kind = "f32" if w.op == "sum_f32" else "bf16"
    check_pair(kind, host, abi.PAIR_OPS[kind](to_device(host)).tolist())


# ---------------------------------------------------------------------------
# the five workload configurations at full size
# ---------------------------------------------------------------------------

_cache = {}


def workload(w):
    if w.name not in _cache:
        _cache.clear()
        _cache[w.name] = inputs.make(w)
    return _cache[w.name]


@pytest.mark.slow
@pytest.mark.parametrize("w", inputs.SMALL + (inputs.CFG2_SUM_F32, inputs.CFG2_SUMSQ_F32, inputs.CFG3_SUM_I32,
                                              inputs.CFG5_SUM_BF16, inputs.CFG5_SUMSQ_BF16),
                         ids=lambda w: w.name)
def test_config_scalar(w):
    host = workload(w)
    got = abi.SCALAR_OPS[w.op](to_device(host)).item()
    check(w.op, host, got)


@pytest.mark.slow
@pytest.mark.parametrize("w", (inputs.CFG4_ROWSUM_WIDE, inputs.CFG4_ROWSUM_SKINNY), ids=lambda w: w.name)
def test_config_rowsum(w):
    host = workload(w)
    got = abi.rdx_rowsum_f32(torch.from_numpy(host).to(DEV)).cpu().numpy().astype(np.float64)
    ref = oracle.rowsum_f32(host)
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    bad = np.nonzero(~(np.abs(got - ref) <= tol))[0]
    assert bad.size == 0, (bad[:5], got[bad[:5]], ref[bad[:5]])


# ---------------------------------------------------------------------------
# row-segmented sum
# ---------------------------------------------------------------------------

SHAPES = [(1, 1), (1, 3), (1, 1000), (3, 5), (7, 3), (31, 4), (33, 8), (33, 255), (100, 16), (100, 33),
          (1000, 256), (1000, 257), (513, 64), (64, 1023), (64, 1024), (64, 1025), (17, 2048), (17, 4099),
          (8, 100_000), (2, 1 << 20), (4097, 128), (50_000, 7), (1, 1 << 22),
          (40, 5121), (300, 6001), (2100, 16385)]   # a block per row, rows of every alignment


@pytest.mark.parametrize("shape", SHAPES, ids=str)
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_rowsum_parity(shape, offset):
    rows, cols = shape
    host = inputs.uniform_f32(rows * cols, seed=rows + cols, lo=-1.0, hi=1.0).reshape(rows, cols)
    x = to_device(host.reshape(-1), offset).view(rows, cols)
    got = abi.rdx_rowsum_f32(x).cpu().numpy().astype(np.float64)
    ref = oracle.rowsum_f32(host)
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    assert np.all(np.abs(got - ref) <= tol)


NARROW_COLS = list(range(1, 66))


@pytest.mark.parametrize("cols", NARROW_COLS)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rowsum_narrow_parity(cols, offset):
    # rows of at most 64 columns are staged through shared memory in tiles of
    # 4096 floats (6144 where a bulk copy stages them); three whole tiles and
    # a ragged fourth of the larger size, at every 4-byte misalignment of the
    # base
    rows = 3 * (6144 // cols) + 5
    host = inputs.uniform_f32(rows * cols, seed=cols * 4 + offset, lo=-1.0, hi=1.0).reshape(rows, cols)
    x = to_device(host.reshape(-1), offset).view(rows, cols)
    got = abi.rdx_rowsum_f32(x).cpu().numpy().astype(np.float64)
    ref = oracle.rowsum_f32(host)
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    bad = np.nonzero(~(np.abs(got - ref) <= tol))[0]
    assert bad.size == 0, (bad[:5], got[bad[:5]], ref[bad[:5]])


@pytest.mark.parametrize("cols", [1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 31, 32, 40, 48, 50, 52, 56, 58, 60, 62, 63, 64])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rowsum_narrow_exact_integers(cols, offset):
    # small integers: every partial sum is exact in float32, so each row sum
    # must equal the integer sum bit for bit (a misplaced, dropped or doubled
    # element changes it); the unaligned bases of 8, 12, 16, ... columns take
    # the rotated or aligned-down reads, and of 2, 4, 6, 8, 16, ... columns
    # the bulk-copy staging, which this checks element by element
    rows = 2 * (6144 // cols) + 3
    vals = (np.arange(rows * cols) * 7919 % 23).astype(np.float32) - 11
    x = to_device(vals, offset).view(rows, cols)
    got = abi.rdx_rowsum_f32(x).cpu().numpy()
    want = vals.reshape(rows, cols).astype(np.int64).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), want)
    assert np.array_equal(oracle.rowsum_f32(vals.reshape(rows, cols)), want.astype(np.float64))


STAGED_COLS = [68, 70, 72, 76, 80, 92, 93, 94, 96, 100, 132, 140, 148, 184, 191, 192, 196, 260, 264, 300, 350, 380,
               400, 409, 410, 512, 513, 600, 1024, 2049, 3072, 3073, 5200, 6000, 6001]


@pytest.mark.parametrize("cols", STAGED_COLS)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rowsum_staged_exact_integers(cols, offset):
    # rows of 65-512 columns whose lanes the short-row kernel would leave
    # half-empty, and every row of 513-6000 columns, go through shared memory
    # in 24 KiB tiles (one bulk copy each) and are summed by groups of 8, 16
    # or 32 lanes: three whole tiles and a ragged fourth, small integers so
    # every row sum is exact, at every 4-byte misalignment of the base; the
    # widths on either side of each rule boundary take other kernels and must
    # agree too
    rows = 3 * (6144 // cols) + 5
    vals = (np.arange(rows * cols) * 7919 % 23).astype(np.float32) - 11
    x = to_device(vals, offset).view(rows, cols)
    got = abi.rdx_rowsum_f32(x).cpu().numpy()
    want = vals.reshape(rows, cols).astype(np.int64).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), want)
    host = inputs.uniform_f32(rows * cols, seed=cols + offset, lo=-1.0, hi=1.0).reshape(rows, cols)
    got = abi.rdx_rowsum_f32(to_device(host.reshape(-1), offset).view(rows, cols)).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - oracle.rowsum_f32(host)) <= 1e-6 * oracle.rowabssum_f32(host) + 1e-30)


@pytest.mark.parametrize("shape", [(100, 257), (64, 1001), (20, 2049), (12, 4095), (40, 5121), (300, 6001),
                                   (2100, 16385)], ids=str)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rowsum_wide_exact_integers(shape, offset):
    # rows of every alignment through the short-row, warp-per-row and
    # block-per-row kernels, with small integers whose sums are exact in
    # float32: each row's head and tail floats must be added exactly once
    rows, cols = shape
    vals = (np.arange(rows * cols) * 7919 % 23).astype(np.float32) - 11
    x = to_device(vals, offset).view(rows, cols)
    got = abi.rdx_rowsum_f32(x).cpu().numpy()
    want = vals.reshape(rows, cols).astype(np.int64).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), want)


@pytest.mark.parametrize("shape", [(100, 257), (64, 1001), (20, 2049), (12, 4095), (40, 5121), (300, 6001)],
                         ids=str)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_rowsum_strided_exact_integers(shape, offset):
    # the same rows read through a leading dimension of cols + 3 (every row at
    # its own alignment): contiguous rows of these widths take the staged
    # kernel, these the short-row, warp-per-row (its edge-float variant from
    # 2048 columns) and block-per-row kernels
    rows, cols = shape
    ld = cols + 3
    vals = (np.arange(rows * ld) * 7919 % 23).astype(np.float32) - 11
    x = to_device(vals, offset).view(rows, ld)[:, :cols]
    got = abi.rdx_rowsum_strided_f32(x).cpu().numpy()
    want = vals.reshape(rows, ld)[:, :cols].astype(np.int64).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), want)


ROWS_STAGED_COLS = [65, 68, 92, 93, 132, 191, 192, 260, 409, 513, 2049, 6000, 6001]


@pytest.mark.parametrize("cols", ROWS_STAGED_COLS)
@pytest.mark.parametrize("pad", [1, 3, 4, 8])
@pytest.mark.parametrize("offset", [0, 1])
def test_rowsum_rows_staged_exact_integers(cols, pad, offset):
    # rows with a leading dimension of cols + pad: where the short-row or
    # warp-per-row kernel would leave load slots empty, each row's 16-byte
    # body is bulk-copied into its own padded slot of shared memory and its
    # edge floats loaded one by one; three whole tiles and a ragged fourth,
    # small integers so every row sum is exact
    ld = cols + pad
    slot = (cols + 4 + 3) // 4 * 4
    rows = 3 * max(1, 6144 // (slot + 28)) + 5
    vals = (np.arange(rows * ld) * 7919 % 23).astype(np.float32) - 11
    x = to_device(vals, offset).view(rows, ld)[:, :cols]
    got = abi.rdx_rowsum_strided_f32(x).cpu().numpy()
    want = vals.reshape(rows, ld)[:, :cols].astype(np.int64).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), want)


@pytest.mark.parametrize("cols", [69, 133, 261, 777])
def test_rows_staged_matches_contiguous_bits(cols):
    # odd widths: the same rows summed contiguously (one bulk copy per tile)
    # and through a leading dimension (one bulk copy per row) take the same
    # lanes and the same order, so their sums agree bit for bit
    rows = 5000
    host = inputs.uniform_f32(rows * cols, seed=cols, lo=-1.0, hi=1.0).reshape(rows, cols)
    contiguous = abi.rdx_rowsum_f32(to_device(host.reshape(-1), 1).view(rows, cols))
    wide = np.zeros((rows, cols + 5), np.float32)
    wide[:, :cols] = host
    strided = abi.rdx_rowsum_strided_f32(to_device(wide.reshape(-1), 2).view(rows, cols + 5)[:, :cols])
    assert torch.equal(contiguous.view(torch.int32), strided.view(torch.int32))
    ref = oracle.rowsum_f32(host)
    assert np.all(np.abs(strided.cpu().numpy().astype(np.float64) - ref) <= 1e-6 * oracle.rowabssum_f32(host) + 1e-30)


def test_rowsum_narrow_deterministic_and_matches_strided():
    for cols in (3, 6, 12, 20, 45):
        x = torch.rand((20_000, cols), device=DEV) * 2 - 1
        a = abi.rdx_rowsum_f32(x)
        for _ in range(3):
            assert torch.equal(abi.rdx_rowsum_f32(x).view(torch.int32), a.view(torch.int32))
        # the same rows read through a leading dimension take another kernel
        wide = torch.zeros((20_000, cols + 5), device=DEV)
        wide[:, :cols] = x
        b = abi.rdx_rowsum_strided_f32(wide[:, :cols])
        host = x.cpu().numpy()
        tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
        assert np.all(np.abs(b.cpu().numpy().astype(np.float64) - a.cpu().numpy().astype(np.float64)) <= 2 * tol)


def test_rowsum_degenerate_shapes():
    out = torch.full((5,), 7.0, device=DEV)
    abi.rdx_rowsum_f32(torch.empty((5, 0), device=DEV), out=out)
    assert out.tolist() == [0.0] * 5
    assert abi.rdx_rowsum_f32(torch.empty((0, 9), device=DEV)).shape == (0,)


def test_rowsum_page_segments():
    # demo 3's per-block outputs are segment sums: B = 256 and 2B = 512
    n = 1 << 18
    x = (np.arange(n) % 7).astype(np.float32)
    period = {256: [762, 771, 766, 768, 770, 765, 774], 512: [1533, 1534, 1535, 1536, 1537, 1538, 1539]}
    xt = torch.from_numpy(x).to(DEV)
    for seg, p in period.items():
        got = abi.rdx_rowsum_f32(xt.view(-1, seg)).cpu().tolist()
        assert got == [p[b % 7] for b in range(n // seg)]
        # a row of B (2B) inputs is exactly the segment a block of versions
        # 1-3 (4-5) reduces: the row sums equal those versions' partials
        for v in ((1, 2, 3) if seg == 256 else (4, 5)):
            assert abi.rdx_ladder_partials_f32(v, xt).cpu().tolist() == got


# ---------------------------------------------------------------------------
# the page's five block reductions: bit-exact against the oracle's restatement
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("version", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("n", [1, 255, 256, 257, 511, 512, 513, 1 << 14, 1 << 18, (1 << 20) + 77])
def test_ladder_bit_exact(version, n):
    host = inputs.normal_f32(n, seed=version)
    got = abi.rdx_ladder_partials_f32(version, torch.from_numpy(host).to(DEV)).cpu().numpy()
    ref = oracle.ladder_partials(version, host)
    assert got.shape == ref.shape
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("version", [1, 2, 3, 4, 5])
def test_ladder_page_worked_example(version):
    for n in (1 << 14, 1 << 18):
        host = (np.arange(n) % 7).astype(np.float32)
        got = abi.rdx_ladder_partials_f32(version, torch.from_numpy(host).to(DEV)).cpu().numpy()
        assert np.array_equal(got, oracle.ladder_partials(version, host))
        assert float(got.astype(np.float64).sum()) == {1 << 14: 49146, 1 << 18: 786429}[n]


@pytest.mark.parametrize("version", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("n", [0, 1, 255, 256, 257, 511, 513, 65537, (1 << 20) + 3, (1 << 24) + 13])
def test_ladder_sum_with_device_finish(version, n):
    # the partials are still the page's, bit for bit; their device-side sum
    # is within the float tolerance of the oracle and repeats bit for bit
    host = inputs.normal_f32(n, seed=version + 50)
    x = torch.from_numpy(host).to(DEV)
    nb, off = abi.rdx_ladder_num_partials(version, n), version % 2  # odd versions: partials 4 bytes off 16
    parts = torch.full((nb + off,), float("nan"), device=DEV)[off:]
    out = abi.rdx_ladder_sum_f32(version, x, partials=parts)
    assert np.array_equal(parts.cpu().numpy().view(np.uint32), oracle.ladder_partials(version, host).view(np.uint32))
    check("sum_f32", host, out.item())
    again = abi.rdx_ladder_sum_f32(version, x, partials=parts)  # same buffers, same bits
    assert again.view(torch.int32).item() == out.view(torch.int32).item()


@pytest.mark.parametrize("version", [1, 2, 3, 4, 5])
def test_ladder_sum_page_worked_example(version):
    # in[i] = i mod 7: every partial and the total are exact integers
    for n, total in ((1 << 14, 49146), (1 << 18, 786429)):
        x = torch.from_numpy((np.arange(n) % 7).astype(np.float32)).to(DEV)
        assert abi.rdx_ladder_sum_f32(version, x).item() == total


def test_ladder_sum_interleaves_with_the_scalar_sums():
    # the ladder's finish and the scalar sums share the stream's completion
    # counter; each launch must leave it ready for the next
    host = inputs.normal_f32((1 << 22) + 5, seed=77)
    x = torch.from_numpy(host).to(DEV)
    outs = []
    for v in (1, 5, 3):
        outs.append(abi.rdx_sum_f32(x))
        outs.append(abi.rdx_ladder_sum_f32(v, x))
    torch.cuda.synchronize()
    for o in outs:
        check("sum_f32", host, o.item())


# ---------------------------------------------------------------------------
# determinism, concurrency, limits, errors
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("op", OPS)
def test_bitwise_deterministic(op):
    x = to_device(host_input(op, (1 << 24) + 13, seed=1))
    fn = abi.SCALAR_OPS[op]
    first = fn(x).clone()
    side = torch.cuda.Stream()
    for i in range(10):
        if i % 2:
            with torch.cuda.stream(side):
                got = fn(x, stream=side)
            side.synchronize()
        else:
            got = fn(x)
        assert torch.equal(got.view(torch.int32 if got.dtype == torch.float32 else torch.int64),
                           first.view(torch.int32 if first.dtype == torch.float32 else torch.int64))


def test_rowsum_deterministic():
    for shape in ((8192, 4096), (1 << 16, 256)):
        x = torch.rand(shape, device=DEV) * 2 - 1
        a = abi.rdx_rowsum_f32(x)
        for _ in range(5):
            assert torch.equal(abi.rdx_rowsum_f32(x).view(torch.int32), a.view(torch.int32))


def test_chained_calls_read_each_others_results():
    # Each call below reads what the call before it wrote, queued back to back
    # on one stream with no host synchronisation: a kernel launched behind
    # another may start early (programmatic dependent launch) and must still
    # see every write of the one ahead.  Small integers keep every result
    # exact, so any stale read shows.
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for seed in range(20):
            host = (np.random.default_rng(seed).integers(-3, 4, size=(1024, 512))).astype(np.float32)
            x = torch.from_numpy(host).to(DEV, non_blocking=False)
            r = abi.rdx_rowsum_f32(x, stream=s)                       # 1024 row sums
            t = abi.rdx_sum_f32(r, stream=s)                          # their total
            m = abi.rdx_max_f32(r, stream=s)                          # their maximum
            rr = abi.rdx_rowsum_f32(r.view(16, 64), stream=s)          # sums of 64 row sums
            t2 = abi.rdx_sum_f32(rr, stream=s)                        # the total again
            z = abi.rdx_sum_i32_i64(r.to(torch.int32), stream=s)     # through a torch kernel
            s.synchronize()
            rows = host.astype(np.int64).sum(axis=1)
            assert np.array_equal(r.cpu().numpy().astype(np.int64), rows)
            assert t.item() == t2.item() == z.item() == rows.sum()
            assert m.item() == rows.max()
            assert np.array_equal(rr.cpu().numpy().astype(np.int64), rows.reshape(16, 64).sum(axis=1))


def test_concurrent_streams():
    hosts = [inputs.normal_f32((1 << 22) + i, seed=10 + i) for i in range(4)]
    devs = [torch.from_numpy(h).to(DEV) for h in hosts]
    streams = [torch.cuda.Stream() for _ in hosts]
    outs = []
    for _ in range(3):
        outs = []
        for x, s in zip(devs, streams):
            with torch.cuda.stream(s):
                outs.append(abi.rdx_sum_f32(x, stream=s))
        torch.cuda.synchronize()
    for h, o in zip(hosts, outs):
        check("sum_f32", h, o.item())


@pytest.mark.slow
def test_largest_sizes_index_math():
    # more than 2^31 elements (int32 and float32, 8 GiB) and more than 2^32
    # bfloat16 elements (8 GiB): all ones, so the sum is n
    n = (1 << 31) + 5
    x = torch.ones(n, dtype=torch.int32, device=DEV)
    assert abi.rdx_sum_i32_i64(x).item() == n
    x = x.view(torch.float32).fill_(1.0)
    assert abs(abi.rdx_sum_f32(x).item() - n) <= 1e-6 * n
    del x
    torch.cuda.empty_cache()
    n = (1 << 32) + 3
    b = torch.ones(n, dtype=torch.bfloat16, device=DEV)
    assert abs(abi.rdx_sum_bf16_f32acc(b).item() - n) <= 4e-6 * n
    del b
    torch.cuda.empty_cache()


def test_workspace_allocation_failure_is_reported(monkeypatch):
    x = torch.ones(1 << 22, device=DEV)
    fresh = torch.cuda.Stream()
    monkeypatch.setenv("RDX_FAULT_ALLOC", "1")
    with pytest.raises(abi.RdxError) as e:
        abi.rdx_sum_f32(x, stream=fresh)
    assert e.value.status == abi.RDX_ERR_ALLOC
    # a one-block launch needs no workspace
    small = abi.rdx_sum_f32(x[:100], stream=fresh)
    fresh.synchronize()
    assert small.item() == 100.0
    monkeypatch.delenv("RDX_FAULT_ALLOC")
    with torch.cuda.stream(fresh):
        got = abi.rdx_sum_f32(x, stream=fresh)
    fresh.synchronize()
    assert got.item() == float(1 << 22)


def test_overlap_and_bad_tensors_rejected():
    x = torch.ones(1000, device=DEV)
    with pytest.raises(abi.RdxError) as e:
        abi.rdx_sum_f32(x[1:], out=x[500])
    assert e.value.status == abi.RDX_ERR_INVALID_ARG
    with pytest.raises(TypeError):
        abi.rdx_sum_f32(x.double())
    with pytest.raises(TypeError):
        abi.rdx_sum_f32(torch.ones(10))
    with pytest.raises(ValueError):
        abi.rdx_sum_f32(torch.ones(10, 10, device=DEV).t())
    assert abi.rdx_sum_f32(x).item() == 1000.0


def test_per_thread_default_stream_gets_a_workspace_per_thread():
    # cudaStreamPerThread (handle 2) is a different stream in every host
    # thread; calls from several threads at once must not share a workspace
    import threading

    lib = abi.load()
    per_thread = 2
    hosts = [inputs.normal_f32((1 << 22) + 31 * i, seed=60 + i) for i in range(4)]
    devs = [torch.from_numpy(h).to(DEV) for h in hosts]
    outs = [[torch.empty((), device=DEV) for _ in range(25)] for _ in hosts]
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(DEV)
            for o in outs[i]:
                st = lib.rdx_sum_f32(devs[i].data_ptr(), devs[i].numel(), o.data_ptr(), per_thread)
                if st != 0:
                    errors.append(st)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(hosts))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for h, row in zip(hosts, outs):
        assert len({o.view(torch.int32).item() for o in row}) == 1  # every call the same bits
        check("sum_f32", h, row[0].item())


def test_host_threads_call_concurrently():
    # ctypes drops the GIL during a call: several host threads enqueue on
    # their own streams at once (per-stream workspaces, no shared state)
    import threading

    hosts = [inputs.normal_f32((1 << 21) + 17 * i, seed=30 + i) for i in range(6)]
    devs = [torch.from_numpy(h).to(DEV) for h in hosts]
    results, errors = {}, []

    def worker(i):
        try:
            torch.cuda.set_device(DEV)
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(20):
                    outs.append(abi.rdx_sum_f32(devs[i], stream=s))
                pair = abi.rdx_sum_sumsq_f32(devs[i], stream=s)
            s.synchronize()
            results[i] = ([o.item() for o in outs], pair.tolist())
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(hosts))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, h in enumerate(hosts):
        sums, pair = results[i]
        assert len(set(sums)) == 1                     # the same bits every time
        check("sum_f32", h, sums[0])
        check("sumsq_f32", h, pair[1])


def test_shutdown_frees_and_calls_reallocate():
    x = torch.from_numpy(inputs.normal_f32((1 << 22) + 3, seed=9)).to(DEV)
    a = abi.rdx_sum_f32(x).clone()
    torch.cuda.synchronize()
    abi.rdx_shutdown()
    b = abi.rdx_sum_f32(x)                     # a fresh workspace, counters zeroed again
    c = abi.rdx_rowsum_f32(x[: 4 * 1000000].view(4, -1))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.isfinite(c).all()
