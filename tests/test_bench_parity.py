"""The bench's own parity check (host logic, no GPU): results within the
tolerance pass, one outside fails, an integer sum must be exact, and steps
that disagree in any bit fail even when each is within the tolerance."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from reduction_rdx_sum_gb300 import inputs  # noqa: E402

W_SUM = inputs.Workload("s", "sum_f32", (8,), "N(0,1)", 1)
W_INT = inputs.Workload("i", "sum_i32", (8,), "Z[-5,5]", 2)
W_ROW = inputs.Workload("r", "rowsum_f32", (3, 4), "U[-1,1)", 3)
OPS = [(W_SUM, None, None, None), (W_INT, None, None, None), (W_ROW, None, None, None)]
REFS = {"s": (10.0, 1e-3), "i": (-7, 0), "r": (np.array([1.0, 2.0, 3.0]), np.array([1e-3, 1e-3, 1e-3]))}


def step(s=10.0, i=-7, r=(1.0, 2.0, 3.0)):
    return [np.array(s, dtype=np.float32), np.array(i, dtype=np.int64), np.array(r, dtype=np.float32)]


def test_results_within_tolerance_and_repeated_pass():
    rep = bench.parity_report(OPS, REFS, [step(10.0005), step(10.0005)], "test")
    assert rep["ok"], rep
    assert rep["s"]["max_err_over_tol"] <= 1.0 and rep["i"]["exact"] and rep["r"]["bitwise_repeat"]


def test_a_float_outside_the_tolerance_fails():
    rep = bench.parity_report(OPS, REFS, [step(10.01)], "test")
    assert not rep["ok"] and not rep["s"]["ok"] and rep["i"]["ok"]


def test_one_row_outside_the_tolerance_fails():
    rep = bench.parity_report(OPS, REFS, [step(r=(1.0, 2.01, 3.0))], "test")
    assert not rep["r"]["ok"] and rep["r"]["max_err_over_tol"] > 1.0


def test_an_inexact_integer_sum_fails():
    rep = bench.parity_report(OPS, REFS, [step(i=-6)], "test")
    assert not rep["ok"] and not rep["i"]["exact"]


def test_steps_that_differ_in_one_bit_fail():
    a = step(10.0)
    b = step(float(np.nextafter(np.float32(10.0), np.float32(11.0))))
    rep = bench.parity_report(OPS, REFS, [a, b], "test")
    assert rep["s"]["max_err_over_tol"] <= 1.0
    assert not rep["s"]["bitwise_repeat"] and not rep["ok"]


def test_nan_fails():
    rep = bench.parity_report(OPS, REFS, [step(float("nan"))], "test")
    assert not rep["s"]["ok"]


def test_back_to_back_order_keeps_shared_arrays_apart():
    """The back-to-back step runs every call once, and two calls on the same
    array (same recipe) have at least L2_APART_BYTES of other calls' reads
    between them, so the second cannot find its input in the L2."""
    by_name = {w.name: w for w in inputs.SUITE}
    order = list(bench.BACK_TO_BACK_ORDER)
    assert sorted(order) == sorted(by_name)
    key = {n: (by_name[n].dist, by_name[n].seed, by_name[n].numel) for n in order}
    for i, a in enumerate(order):
        for j in range(i + 1, len(order)):
            if key[order[j]] == key[a]:
                between = sum(by_name[n].bytes_read for n in order[i + 1:j])
                assert between >= bench.L2_APART_BYTES, (a, order[j], between)
