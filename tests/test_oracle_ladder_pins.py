"""Pins of the numpy restatement of the page's five block-reduction versions
("03_shared_memory_sync_reduction.py", demo 3) to facts outside it: exact
integer segment sums, unit impulses (a wrong index or a dropped term moves or
loses the impulse), the float32 tree error bound, and the page's worked
example.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.ladder import ladder_partials, ladder_segment

VERSIONS = [1, 2, 3, 4, 5]


@pytest.mark.parametrize("version", VERSIONS)
@pytest.mark.parametrize("block", [64, 256])
def test_impulse_lands_in_its_block(version, block):
    seg = ladder_segment(version, block)
    n = 2 * seg + 3                           # two whole blocks and a ragged third
    for pos in range(n):
        x = np.zeros(n, np.float32)
        x[pos] = 1.0
        p = ladder_partials(version, x, block)
        assert p.shape == (3,)
        assert p.tolist() == [1.0 if b == pos // seg else 0.0 for b in range(3)], pos


@pytest.mark.parametrize("version", VERSIONS)
@pytest.mark.parametrize("n", [1, 255, 256, 257, 511, 512, 513, 4096 + 77])
def test_integer_inputs_give_exact_segment_sums(version, n):
    rng = np.random.default_rng(n * 10 + version)
    x = rng.integers(-1000, 1001, n).astype(np.float32)   # all partials stay exact
    seg = ladder_segment(version)
    p = ladder_partials(version, x)
    expect = [float(sum(int(v) for v in x[b * seg:(b + 1) * seg])) for b in range(-(-n // seg))]
    assert p.tolist() == expect


@pytest.mark.parametrize("version", VERSIONS)
def test_float_partials_within_tree_bound(version):
    rng = np.random.default_rng(version)
    x = rng.standard_normal(8 * 512 + 100, dtype=np.float32)
    seg = ladder_segment(version)
    p = ladder_partials(version, x)
    depth = int(np.log2(seg))
    for b, got in enumerate(p):
        s = x[b * seg:(b + 1) * seg]
        ex = sum((Fraction(float(v)) for v in s), Fraction(0))
        a = float(np.abs(s).astype(np.float64).sum())
        # each input passes through at most log2(seg) float32 additions
        assert abs(Fraction(float(got)) - ex) <= Fraction((depth + 1) * U32_SLACK * a)


U32_SLACK = 2.0 ** -24 * 1.01


def test_versions_one_and_two_add_the_same_pairs():
    x = np.random.default_rng(3).standard_normal(256 * 9, dtype=np.float32)
    assert np.array_equal(ladder_partials(1, x), ladder_partials(2, x))


def test_page_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "page_demo3_arange_mod7.txt")) as f:
        lines = [ln.split("#")[0].split() for ln in f if ln.split("#")[0].strip()]
    totals = {int(l[1]): int(l[2]) for l in lines if l[0] == "total"}
    segs = {int(l[1]): [int(v) for v in l[2:]] for l in lines if l[0] == "seg"}
    for n, total in totals.items():
        x = (np.arange(n) % 7).astype(np.float32)
        for v in VERSIONS:
            seg = ladder_segment(v)
            p = ladder_partials(v, x)
            assert p.tolist() == [segs[seg][b % 7] for b in range(n // seg)]
            # the page's check: partials summed in float64 equal the float64 sum
            assert float(p.astype(np.float64).sum()) == total


def test_ladder_agrees_with_rowsum_oracle_on_exact_inputs():
    x = (np.arange(256 * 40) % 13 - 6).astype(np.float32)
    for v in VERSIONS:
        seg = ladder_segment(v)
        assert np.array_equal(ladder_partials(v, x).astype(np.float64), oracle.rowsum_f32(x.reshape(-1, seg)))


def test_bad_arguments():
    with pytest.raises(ValueError):
        ladder_partials(6, np.zeros(4, np.float32))
    with pytest.raises(ValueError):
        ladder_partials(1, np.zeros(4, np.float32), block=96)
    assert ladder_partials(3, np.zeros(0, np.float32)).shape == (0,)


# ---------------------------------------------------------------------------
# the bank-conflict model of demo 1
# ---------------------------------------------------------------------------

def test_bank_rounds_match_the_page(golden_dir):
    from oracle import banks

    with open(os.path.join(golden_dir, "page_demo1_bank_rounds.txt")) as f:
        table = [tuple(int(v) for v in ln.split()) for ln in f if ln.strip() and not ln.startswith("#")]
    assert [p for p, _ in table] == list(range(len(banks.PATTERNS)))
    for p, rounds in table:
        assert banks.wavefronts(banks.indices(p)) == rounds, banks.PATTERNS[p][0]


def test_bank_model_closed_forms():
    from oracle import banks

    for s in range(1, 65):
        # stride s: 32 / (32 / gcd(s, 32)) distinct banks -> gcd(s, 32) words per bank
        words = [s * t for t in range(32)]
        assert banks.wavefronts(words) == math.gcd(s, 32)
    assert banks.wavefronts([5] * 32) == 1
    assert banks.wavefronts([]) == 0
    assert banks.wavefronts([0, 32, 64, 0]) == 3          # repeats of a word do not count twice
