"""Pins of the CPU oracle to facts that do not come from the oracle itself:
closed forms, exact rational sums, the page's worked example and hand-derived
fixtures, brute force over tiny inputs, and invariants.  Each test is chosen so
that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a missing compensation) fails it.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

U64 = 2.0 ** -53   # unit roundoff of float64
U32 = 2.0 ** -24   # unit roundoff of float32


def exact(values) -> Fraction:
    return sum((Fraction(float(v)) for v in values), Fraction(0))


def kahan_bound(abs_sum: float, n: int) -> float:
    # Kahan summation: |E| <= (2u + O(n u^2)) * sum|x_i|  (Higham, Accuracy and
    # Stability of Numerical Algorithms, 2nd ed., eq. 4.9); a slack factor of 2.
    return (4 * U64 + 4 * n * U64 * U64) * abs_sum


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

SIZES = [0, 1, 2, 7, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, (1 << 16) + 3, (1 << 20) + 1]


@pytest.mark.parametrize("n", SIZES)
def test_sum_arange_closed_form(n):
    x = np.arange(n, dtype=np.float32)        # exact in float32 for n <= 2^24
    assert oracle.sum_f32(x) == n * (n - 1) // 2
    assert oracle.abssum_f32(-x) == n * (n - 1) // 2
    assert oracle.sum_f32(-x) == -(n * (n - 1) // 2)


@pytest.mark.parametrize("n", SIZES)
def test_sum_ones_and_alternating(n):
    assert oracle.sum_f32(np.ones(n, np.float32)) == n
    alt = np.where(np.arange(n) % 2 == 0, 1.0, -1.0).astype(np.float32)  # +1, -1, +1, ...
    assert oracle.sum_f32(alt) == n % 2
    assert oracle.sumsq_f32(alt) == n
    assert oracle.abssum_f32(alt) == n


@pytest.mark.parametrize("n", [0, 1, 2, 33, 1000, 1 << 17])
def test_sumsq_arange_closed_form(n):
    x = np.arange(n, dtype=np.float32)
    # sum_{i<n} i^2 = (n-1) n (2n-1) / 6, exact in float64 below 2^53
    assert oracle.sumsq_f32(x) == (n - 1) * n * (2 * n - 1) // 6


@pytest.mark.parametrize("n", [0, 1, 33, 4096, (1 << 20) + 5])
def test_sum_i32_closed_forms(n):
    assert oracle.sum_i32(np.full(n, 7, np.int32)) == 7 * n
    assert oracle.sum_i32(np.full(n, -(2 ** 31), np.int32)) == -(2 ** 31) * n
    assert oracle.sum_i32(np.full(n, 2 ** 31 - 1, np.int32)) == (2 ** 31 - 1) * n
    x = np.arange(n, dtype=np.int64).astype(np.int32)
    assert oracle.sum_i32(x) == n * (n - 1) // 2


def _wrap64(v: int) -> int:
    """v modulo 2^64, as a signed int64."""
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= 1 << 63 else v


@pytest.mark.parametrize("n", [1, 2, 33, 4096])
def test_sum_i64_closed_forms(n):
    assert oracle.sum_i64(np.full(n, -3, np.int64)) == -3 * n
    x = np.arange(n, dtype=np.int64) * (1 << 32)
    assert oracle.sum_i64(x) == (n * (n - 1) // 2) * (1 << 32)
    # addition modulo 2^64: 2^62 four times wraps to 0; INT64_MAX + 1 to INT64_MIN
    assert oracle.sum_i64(np.full(4 * n, 1 << 62, np.int64)) == 0
    assert oracle.sum_i64(np.array([2 ** 63 - 1] + [1] * n, np.int64)) == -(2 ** 63) + n - 1


@pytest.mark.parametrize("n", [1, 5, 64, 1000])
def test_brute_force_i64(n):
    rng = np.random.default_rng(100 + n)
    x = rng.integers(-(2 ** 63), 2 ** 63 - 1, n, dtype=np.int64, endpoint=True)
    assert oracle.sum_i64(x) == _wrap64(sum(int(v) for v in x))
    # the combine of chunk sums is the whole sum: split int32 data anywhere
    z = rng.integers(-(2 ** 31), 2 ** 31, 3 * n + 1, dtype=np.int64).astype(np.int32)
    cuts = sorted(rng.integers(0, z.size + 1, 4))
    parts = [oracle.sum_i32(c) for c in np.split(z, cuts)]
    assert oracle.sum_i64(np.array(parts, np.int64)) == oracle.sum_i32(z)


def test_sum_empty():
    assert oracle.sum_f32(np.zeros(0, np.float32)) == 0.0
    assert oracle.sum_bf16(np.zeros(0, np.uint16)) == 0.0
    assert oracle.sum_i32(np.zeros(0, np.int32)) == 0
    assert oracle.sum_i64(np.zeros(0, np.int64)) == 0
    assert oracle.rowsum_f32(np.zeros((0, 5), np.float32)).shape == (0,)
    assert np.all(oracle.rowsum_f32(np.zeros((4, 0), np.float32)) == 0.0)


# ---------------------------------------------------------------------------
# hand-derived fixtures
# ---------------------------------------------------------------------------

def _read(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return [ln.split("#")[0].strip() for ln in f if ln.split("#")[0].strip()]


def test_tiny_exact_fixture(golden_dir):
    lines = _read(golden_dir, "tiny_exact.txt")
    seen = 0
    for ln in lines:
        kind, rest = ln.split(None, 1)
        if kind == "i32":
            vals, total = rest.split("=")
            x = np.array([int(v) for v in vals.split()], dtype=np.int32)
            assert oracle.sum_i32(x) == int(total)
        else:
            lhs, sq = rest.split(";")
            vals, total = lhs.split("=")
            x = np.array([float(v) for v in vals.split()], dtype=np.float32)
            assert oracle.sum_f32(x) == float(total)
            assert oracle.sumsq_f32(x) == float(sq.split()[1])
            # every permutation-free reordering also reaches it: reverse
            assert oracle.sum_f32(x[::-1].copy()) == float(total)
        seen += 1
    assert seen == 6


def test_bf16_widening_fixture(golden_dir):
    rows = [ln.split() for ln in _read(golden_dir, "bf16_patterns.txt")]
    bits = np.array([int(r[0], 16) for r in rows], dtype=np.uint16)
    vals = [float.fromhex(r[1]) for r in rows]
    assert len(vals) == 14
    for b, v in zip(bits, vals):
        one = np.array([b], np.uint16)
        assert oracle.sum_bf16(one) == v
        assert oracle.abssum_bf16(one) == abs(v)
        assert oracle.sumsq_bf16(one) == v * v
    # all but the two largest magnitudes: the sum is exact in float64
    small = [i for i, v in enumerate(vals) if abs(v) < 1e30]
    assert oracle.sum_bf16(bits[small]) == float(exact(vals[i] for i in small))


def test_page_worked_example_arange_mod7(golden_dir):
    lines = _read(golden_dir, "page_demo3_arange_mod7.txt")
    totals = {int(l.split()[1]): int(l.split()[2]) for l in lines if l.startswith("total")}
    segs = {int(l.split()[1]): [int(v) for v in l.split()[2:]] for l in lines if l.startswith("seg")}
    for n, total in totals.items():
        x = (np.arange(n) % 7).astype(np.float32)
        assert oracle.sum_f32(x) == total
        for seg, period in segs.items():
            rows = oracle.rowsum_f32(x.reshape(-1, seg))
            expect = [period[b % 7] for b in range(n // seg)]
            assert rows.tolist() == expect


# ---------------------------------------------------------------------------
# brute force on tiny inputs against exact rational sums
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 31, 32, 33, 63, 64])
@pytest.mark.parametrize("dist", ["uniform", "normal", "wide", "cancel"])
def test_brute_force_f32(n, dist):
    rng = np.random.default_rng(1000 * n + len(dist))
    if dist == "uniform":
        x = rng.random(n, dtype=np.float32)
    elif dist == "normal":
        x = rng.standard_normal(n, dtype=np.float32)
    elif dist == "wide":   # magnitudes spread over 2^-40 .. 2^40, mixed signs
        x = (rng.standard_normal(n) * 2.0 ** rng.integers(-40, 40, n)).astype(np.float32)
    else:                  # values and their negatives, plus one small term
        h = rng.standard_normal(n, dtype=np.float32)
        x = np.concatenate([h, -h[::-1], np.float32([1e-3])]).astype(np.float32)
    ex = exact(x)
    a = float(sum(abs(Fraction(float(v))) for v in x))
    tol = kahan_bound(a, x.size)
    assert abs(Fraction(oracle.sum_f32(x)) - ex) <= Fraction(tol)
    assert abs(oracle.sum_f32(x) - math.fsum(x.astype(np.float64))) <= tol
    assert abs(oracle.abssum_f32(x) - a) <= tol
    sq = exact(np.float64(v) * np.float64(v) for v in x)   # squares exact in float64
    assert abs(Fraction(oracle.sumsq_f32(x)) - sq) <= Fraction(kahan_bound(float(sq), x.size))


@pytest.mark.parametrize("n", [1, 5, 31, 33, 64])
def test_brute_force_i32(n):
    rng = np.random.default_rng(n)
    x = rng.integers(-(2 ** 31), 2 ** 31, n, dtype=np.int64).astype(np.int32)
    assert oracle.sum_i32(x) == sum(int(v) for v in x)


@pytest.mark.parametrize("n", [1, 7, 33, 64])
def test_brute_force_bf16(n):
    rng = np.random.default_rng(7 + n)
    bits = rng.integers(0, 1 << 16, n, dtype=np.int64).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]              # finite patterns only
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    ex = exact(vals)
    a = float(sum(abs(Fraction(float(v))) for v in vals))
    assert abs(Fraction(oracle.sum_bf16(bits)) - ex) <= Fraction(kahan_bound(a, n))
    sq = exact(np.float64(v) ** 2 for v in vals)
    assert abs(Fraction(oracle.sumsq_bf16(bits)) - sq) <= Fraction(kahan_bound(float(sq), n))


def test_kahan_compensation_is_present():
    # 2^60 followed by 2^16 copies of 16: every 16 is below half an ulp of 2^60
    # in float64 (ulp = 256), so a plain float64 loop returns exactly 2^60 and
    # loses 2^20.  Compensated summation keeps the error within ~2u*sum|x|.
    x = np.concatenate([np.float32([2.0 ** 60]), np.full(1 << 16, 16.0, np.float32)])
    ex = 2 ** 60 + 2 ** 20
    plain = 0.0
    for v in (2.0 ** 60, 16.0):
        plain += v
    assert plain == 2.0 ** 60                       # the effect is real
    assert abs(Fraction(oracle.sum_f32(x)) - ex) <= 1024
    bits = np.concatenate([np.uint16([0x5D80]), np.full(1 << 16, 0x4180, np.uint16)])  # 2^60, 16
    assert abs(Fraction(oracle.sum_bf16(bits)) - ex) <= 1024


# ---------------------------------------------------------------------------
# non-finite values: IEEE propagation as in a plain sum
# ---------------------------------------------------------------------------

def test_nonfinite_propagation():
    inf, nan = np.float32(np.inf), np.float32(np.nan)
    assert oracle.sum_f32(np.float32([1, inf, 3])) == np.inf
    assert oracle.sum_f32(np.float32([-inf, 2])) == -np.inf
    assert math.isnan(oracle.sum_f32(np.float32([inf, 5, -inf])))
    assert math.isnan(oracle.sum_f32(np.float32([1, nan])))
    assert oracle.sumsq_f32(np.float32([-inf, 1])) == np.inf
    assert oracle.sum_bf16(np.uint16([0x3F80, 0x7F80])) == np.inf   # 1 + (+Inf)
    assert math.isnan(oracle.sum_bf16(np.uint16([0x7FC0])))         # NaN


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def test_permutation_and_concatenation_invariants():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(100_003, dtype=np.float32)
    a = oracle.abssum_f32(x)
    p = rng.permutation(x.size)
    assert abs(oracle.sum_f32(x[p]) - oracle.sum_f32(x)) <= 2 * kahan_bound(a, x.size)
    xi = rng.integers(-(2 ** 31), 2 ** 31, 50_001, dtype=np.int64).astype(np.int32)
    assert oracle.sum_i32(xi) == oracle.sum_i32(xi[:20_000]) + oracle.sum_i32(xi[20_000:])


def test_rowsum_rows_and_orientation():
    rng = np.random.default_rng(11)
    m = rng.standard_normal((3, 5), dtype=np.float32)
    rows = oracle.rowsum_f32(m)
    for r in range(3):
        assert abs(rows[r] - math.fsum(m[r].astype(np.float64))) <= kahan_bound(float(np.abs(m[r]).sum()), 5)
    # a transposed operand would give column sums: they differ here
    assert not np.allclose(rows, oracle.rowsum_f32(np.ascontiguousarray(m.T))[:3])
    # one row is the plain sum; row sums add up to the total
    x = rng.standard_normal(4097, dtype=np.float32)
    assert oracle.rowsum_f32(x.reshape(1, -1))[0] == oracle.sum_f32(x)
    ab = oracle.rowabssum_f32(m)
    assert np.allclose(ab, np.abs(m).astype(np.float64).sum(axis=1), rtol=1e-15, atol=0)
    # a single non-zero lands in its own row only
    for pos in range(15):
        e = np.zeros(15, np.float32)
        e[pos] = 1.0
        out = oracle.rowsum_f32(e.reshape(3, 5))
        assert out.tolist() == [1.0 if r == pos // 5 else 0.0 for r in range(3)]


# ---------------------------------------------------------------------------
# maximum
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 31, 33, 1000, (1 << 16) + 3])
def test_max_closed_forms_and_impulses(n):
    assert oracle.max_f32(np.arange(n, dtype=np.float32)) == n - 1
    assert oracle.max_f32(-np.arange(n, dtype=np.float32)) == 0.0
    assert oracle.max_i32(np.arange(n, dtype=np.int32) - n) == -1
    for pos in sorted({0, n // 3, n - 1}):
        x = np.full(n, -5.0, np.float32)
        x[pos] = 7.5
        assert oracle.max_f32(x) == 7.5
        z = np.full(n, -(2 ** 31), np.int32)
        z[pos] = 2 ** 31 - 1
        assert oracle.max_i32(z) == 2 ** 31 - 1


def test_max_special_values():
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    assert oracle.max_f32(np.zeros(0, np.float32)) == -np.inf
    assert oracle.max_f32(np.float32([nan, nan])) == -np.inf
    assert oracle.max_f32(np.float32([nan, 1, nan, -3])) == 1.0      # NaN never wins
    assert oracle.max_f32(np.float32([-inf, -1e30])) == np.float32(-1e30)
    assert oracle.max_f32(np.float32([1, inf, 2])) == np.inf
    assert oracle.max_i32(np.zeros(0, np.int32)) == -(2 ** 31)


@pytest.mark.parametrize("n", [1, 7, 64])
def test_max_brute_force(n):
    rng = np.random.default_rng(40 + n)
    x = (rng.standard_normal(n) * 2.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    assert oracle.max_f32(x) == max(float(v) for v in x)
    z = rng.integers(-(2 ** 31), 2 ** 31, n, dtype=np.int64).astype(np.int32)
    assert oracle.max_i32(z) == max(int(v) for v in z)
