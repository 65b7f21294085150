import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (GiB inputs)")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_sessionfinish(session, exitstatus):
    """With RDX_LIBRARY naming the checked build, the run fails if any kernel
    access fell outside its buffer."""
    if not os.environ.get("RDX_LIBRARY"):
        return
    from reduction_rdx_sum_gb300 import abi

    if abi._lib is None or not abi.rdx_debug_build():
        return
    n = abi.rdx_debug_violations()
    print(f"\nchecked build: {n} out-of-range accesses")
    if n != 0:
        session.exitstatus = 1
