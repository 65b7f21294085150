"""The seeded input generator: reproducible, independent of the thread count,
the stated ranges, and the float32 -> bfloat16 rounding."""
import numpy as np
import pytest
import torch

from reduction_rdx_sum_gb300 import inputs


def test_reproducible_and_seed_dependent():
    a = inputs.normal_f32(3 * inputs.CHUNK + 17, seed=1)
    b = inputs.normal_f32(3 * inputs.CHUNK + 17, seed=1)
    c = inputs.normal_f32(3 * inputs.CHUNK + 17, seed=2)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)


def test_prefix_stable_and_thread_count_free(monkeypatch):
    long = inputs.uniform_f32(2 * inputs.CHUNK + 5, seed=0)
    short = inputs.uniform_f32(inputs.CHUNK + 3, seed=0)
    assert np.array_equal(long[: short.size], short)
    monkeypatch.setattr(inputs, "_threads", lambda: 1)
    assert np.array_equal(inputs.uniform_f32(2 * inputs.CHUNK + 5, seed=0), long)


def test_ranges():
    u = inputs.uniform_f32(1 << 20, seed=0)
    assert u.min() >= 0.0 and u.max() < 1.0
    v = inputs.uniform_f32(1 << 20, seed=3, lo=-1.0, hi=1.0)
    assert v.min() >= -1.0 and v.max() < 1.0 and v.min() < -0.99 and v.max() > 0.99
    z = inputs.integers_i32(1 << 20, seed=0, lo=-1000, hi=1000)
    assert z.dtype == np.int32 and z.min() == -1000 and z.max() == 1000
    g = inputs.normal_f32(1 << 20, seed=1)
    assert abs(float(g.mean())) < 0.01 and abs(float(g.std()) - 1.0) < 0.01


def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100_000, dtype=np.float32),
        # exact ties (the 16 dropped bits are 0x8000) on finite upper halves, both signs
        (((rng.integers(0, 0x7F80, 1000, dtype=np.uint32) | (rng.integers(0, 2, 1000, dtype=np.uint32) << 15)) << 16)
         | 0x8000).view(np.float32),
        np.float32([0.0, -0.0, 1.0, 3.4e38, -3.4e38, 1e-40]),
    ]).astype(np.float32)
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_workload_table():
    assert inputs.CFG2_SUM_F32.shape == ((1 << 24) + 13,)
    assert inputs.CFG4_ROWSUM_WIDE.bytes_read == 1 << 30
    assert inputs.CFG4_ROWSUM_SKINNY.bytes_read == 1 << 30
    assert inputs.CFG5_SUM_BF16.bytes_read == 2 * ((1 << 30) + 7)
    small = inputs.make(inputs.CFG1_SUM_I32)
    assert small.dtype == np.int32 and small.shape == (1 << 20,)
    assert small.min() == -1000 and small.max() == 1000


@pytest.mark.parametrize("n", [0, 1, inputs.CHUNK - 1, inputs.CHUNK + 1])
def test_edge_sizes(n):
    assert inputs.normal_bf16_bits(n, seed=4).shape == (n,)
    assert inputs.integers_i32(n, seed=2, lo=-5, hi=5).shape == (n,)
