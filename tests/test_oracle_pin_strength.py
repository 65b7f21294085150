"""The pins catch planted mistakes.  Each mutant below is a plausible slip in
the oracle (a dropped term, a skipped element, a wrong sign, index, shift or
stride, an inverted comparison); it is compiled from a modified copy of
oracle.c (or, for the ladder, a modified copy of ladder.py) and must fail at
least one pin.  Mistakes are planted in the oracle only, on the CPU."""
import importlib.util
import os
import subprocess
import sys
import types

import numpy as np
import pytest

import oracle
import test_oracle_ladder_pins as lp
import test_oracle_pins as op

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")

C_MUTANTS = [
    ("no compensation", "k->c = (t - k->s) - y;", "k->c = 0.0;"),
    ("compensation sign", "double y = v - k->c;", "double y = v + k->c;"),
    ("skips the first float", "for (int64_t i = 0; i < n; ++i) kahan_add(&k, (double)x[i]);",
     "for (int64_t i = 1; i < n; ++i) kahan_add(&k, (double)x[i]);"),
    ("drops the last square", "    for (int64_t i = 0; i < n; ++i) {\n        double v = (double)x[i];\n        kahan_add(&k, v * v);",
     "    for (int64_t i = 0; i + 1 < n; ++i) {\n        double v = (double)x[i];\n        kahan_add(&k, v * v);"),
    ("square without the square", "        double v = (double)x[i];\n        kahan_add(&k, v * v);",
     "        double v = (double)x[i];\n        kahan_add(&k, v * fabs(v));"),
    ("bf16 widened by 15 bits", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("int sum in 32 bits", "for (int64_t i = 0; i < n; ++i) s += (uint64_t)(int64_t)x[i];",
     "for (int64_t i = 0; i < n; ++i) s = (uint32_t)(s + (uint64_t)(int64_t)x[i]);"),
    ("int64 sum drops the last", "    for (int64_t i = 0; i < n; ++i) s += (uint64_t)x[i];",
     "    for (int64_t i = 0; i + 1 < n; ++i) s += (uint64_t)x[i];"),
    ("int64 sum saturates instead of wrapping", "    for (int64_t i = 0; i < n; ++i) s += (uint64_t)x[i];\n    return from_twos_complement(s);",
     "    long double t = 0;\n    for (int64_t i = 0; i < n; ++i) t += (long double)x[i];\n    (void)s;\n    return t > 9.2e18L ? INT64_MAX : t < -9.2e18L ? INT64_MIN : (int64_t)t;"),
    ("row stride off by one", "const float* row = x + r * cols;\n        kahan_acc k;\n        kahan_init(&k);\n        for (int64_t j = 0; j < cols; ++j) kahan_add(&k, (double)row[j]);",
     "const float* row = x + r * (cols + (r > 0));\n        kahan_acc k;\n        kahan_init(&k);\n        for (int64_t j = 0; j < cols; ++j) kahan_add(&k, (double)row[j]);"),
    ("rows summed as columns", "for (int64_t j = 0; j < cols; ++j) kahan_add(&k, (double)row[j]);\n        out[r] = kahan_result(&k);",
     "for (int64_t j = 0; j < cols && j < rows; ++j) kahan_add(&k, (double)x[j * cols + r]);\n        out[r] = kahan_result(&k);"),
    ("abs dropped", "for (int64_t i = 0; i < n; ++i) kahan_add(&k, fabs((double)x[i]));",
     "for (int64_t i = 0; i < n; ++i) kahan_add(&k, ((double)x[i]));"),
    ("non-finite terms lost", "        k->nonfinite += v;\n        return;", "        return;"),
    ("max keeps the smallest", "        if (x[i] > m) m = x[i];\n    return m;\n}\n\nint32_t",
     "        if (x[i] < m || m == -INFINITY) m = x[i];\n    return m;\n}\n\nint32_t"),
    ("max skips the last", "int32_t oracle_max_i32(const int32_t* x, int64_t n) {\n    int32_t m = INT32_MIN;\n    for (int64_t i = 0; i < n; ++i)",
     "int32_t oracle_max_i32(const int32_t* x, int64_t n) {\n    int32_t m = INT32_MIN;\n    for (int64_t i = 0; i + 1 < n; ++i)"),
]


def pin_battery():
    """Run the C-oracle pins; return the names of those that fail."""
    checks = [
        ("arange", lambda: [op.test_sum_arange_closed_form(n) for n in (1, 33, 1000, (1 << 16) + 3)]),
        ("ones/alternating", lambda: [op.test_sum_ones_and_alternating(n) for n in (1, 2, 33, 513)]),
        ("sumsq closed form", lambda: [op.test_sumsq_arange_closed_form(n) for n in (2, 33, 1000)]),
        ("i32 closed forms", lambda: [op.test_sum_i32_closed_forms(n) for n in (1, 33, 4096)]),
        ("tiny exact", lambda: op.test_tiny_exact_fixture(GOLDEN)),
        ("bf16 fixture", lambda: op.test_bf16_widening_fixture(GOLDEN)),
        ("page example", lambda: op.test_page_worked_example_arange_mod7(GOLDEN)),
        ("brute force f32", lambda: [op.test_brute_force_f32(n, d) for n in (7, 33, 64)
                                     for d in ("uniform", "normal", "wide", "cancel")]),
        ("brute force i32", lambda: [op.test_brute_force_i32(n) for n in (5, 64)]),
        ("i64 closed forms", lambda: [op.test_sum_i64_closed_forms(n) for n in (1, 33)]),
        ("brute force i64", lambda: [op.test_brute_force_i64(n) for n in (5, 64)]),
        ("brute force bf16", lambda: [op.test_brute_force_bf16(n) for n in (7, 64)]),
        ("compensation", op.test_kahan_compensation_is_present),
        ("non-finite", op.test_nonfinite_propagation),
        ("rows", op.test_rowsum_rows_and_orientation),
        ("max", lambda: [op.test_max_closed_forms_and_impulses(n) for n in (2, 33, 1000)]),
        ("max special", op.test_max_special_values),
        ("max brute force", lambda: [op.test_max_brute_force(n) for n in (7, 64)]),
    ]
    failed = []
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, TypeError, ValueError, OverflowError):
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_the_battery():
    oracle.use_library(None)
    assert pin_battery() == []


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_mutant_is_caught(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert old in src, f"mutation site not found: {name}"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    str(mutant), "-o", str(lib), "-lm"], check=True)
    try:
        oracle.use_library(str(lib))
        failed = pin_battery()
    finally:
        oracle.use_library(None)
    assert failed, f"no pin caught the mutant '{name}'"


LADDER_MUTANTS = [
    ("sequential tail off by one", "sdata[:, :s] = sdata[:, :s] + sdata[:, s : 2 * s]",
     "sdata[:, :s] = sdata[:, :s] + sdata[:, s - 1 : 2 * s - 1]"),
    ("interleaved stride", "tid = np.arange(0, block, 2 * s)", "tid = np.arange(0, block, s)[: block // (2 * s)]"),
    ("strided index", "index = 2 * s * np.arange(block)", "index = s * np.arange(block)"),
    ("first add drops the second half", "sdata = seg[:, :block] + seg[:, block:]\n    _sequential_tail(sdata, block)\n",
     "sdata = seg[:, :block] + 0 * seg[:, block:]\n    _sequential_tail(sdata, block)\n"),
    ("shuffle reads the wrong lane", "received[:, : 32 - off] = val[:, off:32]",
     "received[:, : 32 - off] = val[:, off - 1:31]"),
    ("warp stage skips the upper half", "val = sdata[:, 0:32] + sdata[:, 32:64]", "val = sdata[:, 0:32] + 0 * sdata[:, 32:64]"),
    ("tail not masked to zero", "buf = np.zeros(nb * seg, dtype=np.float32)", "buf = np.ones(nb * seg, dtype=np.float32)"),
]


def ladder_battery():
    checks = [
        ("impulses", lambda: [lp.test_impulse_lands_in_its_block(v, b) for v in range(1, 6) for b in (64, 256)]),
        ("integer segments", lambda: [lp.test_integer_inputs_give_exact_segment_sums(v, n) for v in range(1, 6)
                                      for n in (257, 513, 4096 + 77)]),
        ("tree bound", lambda: [lp.test_float_partials_within_tree_bound(v) for v in range(1, 6)]),
        ("page example", lambda: lp.test_page_worked_example(GOLDEN)),
        ("versions 1 and 2", lp.test_versions_one_and_two_add_the_same_pairs),
    ]
    failed = []
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, IndexError, ValueError):
            failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", LADDER_MUTANTS, ids=[m[0] for m in LADDER_MUTANTS])
def test_ladder_mutant_is_caught(monkeypatch, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "ladder.py")).read()
    assert old in src, f"mutation site not found: {name}"
    mod = types.ModuleType("ladder_mutant")
    exec(compile(src.replace(old, new, 1), "ladder_mutant.py", "exec"), mod.__dict__)
    monkeypatch.setattr(lp, "ladder_partials", mod.ladder_partials)
    monkeypatch.setattr(lp, "ladder_segment", mod.ladder_segment)
    monkeypatch.setattr(oracle, "ladder_partials", mod.ladder_partials)
    assert ladder_battery(), f"no pin caught the ladder mutant '{name}'"
