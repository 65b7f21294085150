"""rdx_max_f32 / rdx_max_i32 against the oracle's maximum (the page's
atomic_max rule folded from -Inf): exact equality, every size class, the
maximum placed at the head, the middle and the tail, misaligned bases,
NaN and empty inputs, and the caller-owned workspace path."""
import math

import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, inputs

from test_parity_gpu import DEV, SIZES, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from reduction_rdx_sum_gb300 import build
    build.build()
    oracle.build()
    abi.load()
    torch.cuda.set_device(DEV)


@pytest.mark.parametrize("n", SIZES)
def test_max_parity(n):
    x = inputs.normal_f32(n, seed=n % 53)
    assert abi.rdx_max_f32(to_device(x)).item() == oracle.max_f32(x)
    z = inputs.integers_i32(n, seed=n % 53, lo=-(2 ** 31), hi=2 ** 31 - 1)
    assert abi.rdx_max_i32(to_device(z)).item() == oracle.max_i32(z)


@pytest.mark.parametrize("n", [1, 5, 4097, (1 << 20) + 3, (1 << 24) + 13])
def test_max_impulse_anywhere_and_misaligned(n):
    for pos in sorted(p for p in {0, 1, n // 2, n - 2, n - 1} if 0 <= p < n):
        x = np.full(n, -3.0, np.float32)
        x[pos] = 1.5
        for offset in (0, 1, 3):
            assert abi.rdx_max_f32(to_device(x, offset)).item() == 1.5
        z = np.full(n, -7, np.int32)
        z[pos] = 9
        assert abi.rdx_max_i32(to_device(z, 1)).item() == 9


def test_max_special_values():
    assert abi.rdx_max_f32(torch.empty(0, device=DEV)).item() == -math.inf
    assert abi.rdx_max_i32(torch.empty(0, dtype=torch.int32, device=DEV)).item() == -(2 ** 31)
    x = torch.full((100_003,), math.nan, device=DEV)
    assert abi.rdx_max_f32(x).item() == -math.inf                     # all NaN
    x[77] = -2.0
    x[5000] = -1.0
    assert abi.rdx_max_f32(x).item() == -1.0                           # NaNs never win
    x[99_999] = math.inf
    assert abi.rdx_max_f32(x).item() == math.inf


def test_max_through_workspace_entry():
    ws = torch.zeros(abi.rdx_workspace_bytes(), dtype=torch.uint8, device=DEV)
    x = inputs.normal_f32((1 << 22) + 1, seed=8)
    z = inputs.integers_i32((1 << 22) + 1, seed=8, lo=-(2 ** 31), hi=2 ** 31 - 1)
    assert abi.rdx_reduce_ws("max_f32", to_device(x), ws).item() == oracle.max_f32(x)
    assert abi.rdx_reduce_ws("max_i32", to_device(z), ws).item() == oracle.max_i32(z)


def test_max_word_keys_order_like_floats():
    # The float maximum finishes through an unsigned key per block total
    # (non-negative values with the sign bit set, negative ones inverted).
    # Inputs of many blocks whose maximum is negative, tiny, a zero of either
    # sign, or -Inf, and maxima that differ from the runner-up in the last bit.
    n = (1 << 20) + 5
    cases = {
        "all negative": np.full(n, -5.0, np.float32),
        "negative, tiny": np.full(n, -1e-30, np.float32),
        "zeros of both signs": np.where(np.arange(n) % 2 == 0, np.float32(-0.0), np.float32(0.0)),
        "only -0": np.full(n, -0.0, np.float32),
        "only -Inf": np.full(n, -np.inf, np.float32),
        "subnormals": np.full(n, -1e-44, np.float32),
    }
    cases["negative, tiny"][n // 3] = np.float32(-1e-31)
    cases["subnormals"][n - 7] = np.float32(1e-45)
    adjacent = np.full(n, np.float32(1.0), np.float32)
    adjacent[n // 2] = np.nextafter(np.float32(1.0), np.float32(2.0))
    cases["adjacent floats"] = adjacent
    nadj = np.full(n, np.float32(-1.0), np.float32)
    nadj[12345] = np.nextafter(np.float32(-1.0), np.float32(0.0))
    cases["adjacent negatives"] = nadj
    for name, x in cases.items():
        got = abi.rdx_max_f32(to_device(x)).item()
        assert got == oracle.max_f32(x), name                       # -0 == +0 for a zero maximum
    # two calls in a row on one stream: the word is left clear for the next
    assert abi.rdx_max_f32(to_device(cases["all negative"])).item() == -5.0
    assert abi.rdx_max_f32(to_device(cases["only -Inf"])).item() == -math.inf
