"""The split sum's exchange over NCCL on the GPU, with one rank.

Every call of this test suite gets one GPU, so the NCCL path runs with a
world of one: reduction_rdx_sum_gb300.shard.sharded_reduce takes the rank's
chunk (the whole array), its partial on the device, an NCCL all-gather of one
partial into a device array, and the rank-order combine.  Nothing waits on
another rank.  The result must equal the one-chunk emulation bit for bit and
the oracle (int exact, floats in tolerance).  The bench's own sharded
measurement then runs on the same process group, on small workloads of the
bench's recipes, and must report every result matching the oracle.  Runs in
a child process, so the test session keeps no process group.
"""
import os
import socket
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, ROOT)
import numpy as np, torch, torch.distributed as dist
import oracle
from reduction_rdx_sum_gb300 import build, inputs, shard
build.build(); oracle.build()
torch.cuda.set_device(0)
dist.init_process_group("nccl", rank=0, world_size=1, init_method=f"tcp://127.0.0.1:{PORT}")
dev = torch.device("cuda:0")
cases = {"sum_f32": inputs.normal_f32((1 << 22) + 13, seed=1),
         "sum_i32": inputs.integers_i32((1 << 22) + 5, seed=2, lo=-(2 ** 31), hi=2 ** 31 - 1),
         "sum_sumsq_bf16": inputs.normal_bf16_bits((1 << 23) + 7, seed=4)}
for op, host in cases.items():
    t = torch.from_numpy(host.view(np.int16) if host.dtype == np.uint16 else host).to(dev)
    world, rank = dist.get_world_size(), dist.get_rank()
    got = shard.sharded_reduce(op, shard.local_chunk(op, t, world, rank))
    emu = shard.emulate(op, t, world)
    torch.cuda.synchronize()
    assert got.cpu().numpy().tobytes() == emu.cpu().numpy().tobytes(), op
    if op == "sum_i32":
        assert got.item() == oracle.sum_i32(host)
    elif op == "sum_f32":
        assert abs(got.item() - oracle.sum_f32(host)) <= 1e-6 * oracle.abssum_f32(host)
    else:
        v = got.cpu().numpy().astype(np.float64)
        assert abs(v[0] - oracle.sum_bf16(host)) <= 4e-6 * oracle.abssum_bf16(host)
        q = oracle.sumsq_bf16(host)
        assert abs(v[1] - q) <= 4e-6 * q

# the bench's own sharded measurement on the same process group, on small
# workloads of the same recipes
import bench
from reduction_rdx_sum_gb300.runop import L2Flush

class Small:
    torch = torch
    stream = torch.cuda.current_stream(dev)
    def __init__(self):
        self.flush = L2Flush(dev, 64 << 20)
        self.dev_arrays = {}
    @staticmethod
    def key(w):
        return (w.dist, w.seed, w.numel)
    def event(self):
        return torch.cuda.Event(enable_timing=True)

small = [inputs.Workload("s_bf16", "sum_bf16", ((1 << 22) + 7,), "N(0,1)->bf16", 4),
         inputs.Workload("s_i32", "sum_i32", ((1 << 22) + 3,), "Z[-1048576,1048576]", 2)]
g = Small()
arrays = {}
for w in small:
    h = inputs.make(w).reshape(-1)
    arrays[w.name] = h
    g.dev_arrays[g.key(w)] = torch.from_numpy(h.view(np.int16) if h.dtype == np.uint16 else h).to(dev)
refs = {"s_bf16": (oracle.sum_bf16(arrays["s_bf16"]), 4e-6 * oracle.abssum_bf16(arrays["s_bf16"]) + 1e-30),
        "s_i32": (oracle.sum_i32(arrays["s_i32"]), 0)}
res = bench.measure_sharded(g, refs, dist.get_world_size(), dist.get_rank(), 3, workloads=small)
assert set(res) == {"s_bf16_split1", "s_i32_split1"}, res
assert all(v["parity_ok"] and v["ranks"] == 1 and v["us"] > 0 for v in res.values()), res
dist.destroy_process_group()
print("nccl split ok")
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_sharded_reduce_over_nccl_with_one_rank():
    code = CHILD.replace("ROOT", repr(ROOT)).replace("{PORT}", str(_free_port()))
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "nccl split ok" in r.stdout
