"""The bank-conflict probe of the page's demo 1 on the GPU against the page's
bank model (oracle.banks): clock cycles per shared load grow with the rounds
the model predicts, and conflict-free patterns cost what stride 1 costs."""
import pytest
import torch

from oracle import banks
from reduction_rdx_sum_gb300 import abi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cycles():
    from reduction_rdx_sum_gb300 import build
    build.build()
    abi.load()
    torch.cuda.set_device(0)
    return {p: min(abi.rdx_bank_probe(p, iters=512) for _ in range(3)) for p in range(len(banks.PATTERNS))}


def test_cycles_follow_the_model(cycles):
    rounds = {p: banks.wavefronts(banks.indices(p)) for p in cycles}
    base = cycles[0]
    # conflict-free patterns (odd strides, broadcast, pairs) cost what stride 1 costs
    for p, c in cycles.items():
        if rounds[p] == 1:
            assert c <= 1.1 * base, (banks.PATTERNS[p][0], c, base)
    # each doubling of the rounds doubles the cost once the rounds, not the
    # issue rate, set it (one warp: about two cycles per wavefront)
    by_rounds = {rounds[p]: cycles[p] for p in range(6)}          # strides 1 .. 32
    for w in (4, 8, 16):
        assert 1.6 <= by_rounds[2 * w] / by_rounds[w] <= 2.2, (w, by_rounds)
    assert by_rounds[4] >= 1.5 * base
    assert by_rounds[32] >= 8 * base
    strides = [cycles[p] for p in range(6)]
    assert all(b >= 0.95 * a for a, b in zip(strides, strides[1:]))


def test_probe_rejects_bad_arguments():
    with pytest.raises(abi.RdxError):
        abi.rdx_bank_probe(10)
    with pytest.raises(abi.RdxError):
        abi.rdx_bank_probe(0, iters=0)
