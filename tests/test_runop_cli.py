"""The single-op driver's command line, on the host (no GPU needed to reject
bad arguments)."""
import pytest

from reduction_rdx_sum_gb300 import inputs, runop


def test_needs_exactly_one_of_op_and_config():
    with pytest.raises(SystemExit):
        runop.main([])
    with pytest.raises(SystemExit):
        runop.main(["--op", "sum_f32", "--config", "c2_sum_f32"])
    with pytest.raises(SystemExit):
        runop.main(["--config", "no_such_workload"])


def test_every_workload_has_an_entry_point():
    for w in inputs.ALL:
        assert callable(runop.entry(w.op))


def test_negative_offset_rejected():
    with pytest.raises(SystemExit):
        runop.main(["--op", "rowsum_f32", "--offset", "-1"])


def test_leading_dimension_only_for_row_sums_and_not_below_cols():
    with pytest.raises(SystemExit):
        runop.main(["--op", "sum_f32", "--ld", "10"])
    with pytest.raises(SystemExit):
        runop.main(["--op", "rowsum_f32", "--rows", "4", "--cols", "8", "--ld", "7"])
