"""The bounded wait of the narrow-row kernel's bulk-copy staging.

Rows of fewer than 64 columns whose shared-memory reads would share a bank
(16 columns 4 bytes off 16-byte alignment, for one) arrive tile by tile by
one bulk copy each, and the block waits on a shared-memory barrier for the
copy's bytes.  That wait is bounded: the test hook arms one tile's barrier
for 16 bytes more than its copy brings, so nothing completes it.  The wait
must give up after about a second, count one timeout (rdx_wait_timeouts),
leave its rows unwritten and leave the context usable: the next calls run
and match the oracle, and the normal calls count no timeout.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, inputs

from test_parity_gpu import DEV, to_device

pytestmark = pytest.mark.gpu


def _skewed_rows(rows, cols, seed):
    host = inputs.uniform_f32(rows * cols, seed=seed, lo=-1.0, hi=1.0).reshape(rows, cols)
    return host, to_device(host.reshape(-1), 1).view(rows, cols)   # 4 bytes off 16-byte alignment


def _check_rows(host, got):
    ref = oracle.rowsum_f32(host)
    assert np.all(np.abs(got.cpu().numpy().astype(np.float64) - ref) <= 1e-6 * oracle.rowabssum_f32(host) + 1e-30)


def test_bulk_staged_rows_count_no_timeout():
    abi.rdx_wait_timeouts(reset=True)
    for cols in (4, 8, 16, 24, 40):
        host, x = _skewed_rows(100_003, cols, cols)
        _check_rows(host, abi.rdx_rowsum_f32(x))
    assert abi.rdx_wait_timeouts() == 0


def test_a_wait_that_cannot_complete_gives_up_and_is_counted():
    abi.rdx_wait_timeouts(reset=True)
    x = torch.arange(100 * 16, dtype=torch.float32, device=DEV).view(100, 16)
    out = torch.full((100,), -7.0, device=DEV)
    t0 = time.monotonic()
    abi.rdx_debug_stage_timeout(x, out)
    assert abi.rdx_wait_timeouts() == 1          # synchronizes: the block has given up and exited
    elapsed = time.monotonic() - t0
    assert 0.9 < elapsed < 30.0, elapsed          # one bounded wait of a second, then a second one
    assert torch.all(out == -7.0)                 # its rows were not written
    # the context is still usable: real calls run, match the oracle, count nothing more
    host, xs = _skewed_rows(50_001, 16, 3)
    _check_rows(host, abi.rdx_rowsum_f32(xs))
    assert abi.rdx_sum_f32(x.reshape(-1)).item() == float(sum(range(1600)))
    assert abi.rdx_wait_timeouts(reset=True) == 1
    assert abi.rdx_wait_timeouts() == 0
