"""Caller-owned workspaces (rdx_reduce_ws), rows with a leading dimension
(rdx_rowsum_strided_f32) and the split-row path for few, very long rows, each
against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from reduction_rdx_sum_gb300 import abi, inputs

from test_parity_gpu import DEV, VEC, check, host_input, to_device

pytestmark = pytest.mark.gpu

NAMED = {"sum_f32": abi.rdx_sum_f32, "sumsq_f32": abi.rdx_sumsq_f32, "sum_bf16": abi.rdx_sum_bf16_f32acc,
         "sumsq_bf16": abi.rdx_sumsq_bf16_f32acc, "sum_i32": abi.rdx_sum_i32_i64,
         "sum_sumsq_f32": abi.rdx_sum_sumsq_f32, "sum_sumsq_bf16": abi.rdx_sum_sumsq_bf16_f32acc}
SOURCE = {"sum_sumsq_f32": "sum_f32", "sum_sumsq_bf16": "sum_bf16"}


@pytest.fixture(scope="module")
def workspace():
    from reduction_rdx_sum_gb300 import build
    build.build()
    oracle.build()
    abi.load()
    torch.cuda.set_device(DEV)
    return torch.zeros(abi.rdx_workspace_bytes(), dtype=torch.uint8, device=DEV)


def as_bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


@pytest.mark.parametrize("op", list(NAMED))
@pytest.mark.parametrize("n", [0, 1, 7, 1000, 4097, (1 << 20) + 3, (1 << 24) + 13])
def test_reduce_ws_matches_named_entry_point(workspace, op, n):
    src = SOURCE.get(op, op)
    host = host_input(src, n, seed=n % 31)
    x = to_device(host)
    got = abi.rdx_reduce_ws(op, x, workspace)
    ref = NAMED[op](x)
    assert torch.equal(as_bits(got), as_bits(ref))      # same kernel, same tiling
    if op in SOURCE:
        s_op, q_op = (("sum_f32", "sumsq_f32") if op.endswith("f32") else ("sum_bf16", "sumsq_bf16"))
        g = got.tolist()
        check(s_op, host, g[0])
        check(q_op, host, g[1])
    else:
        check(op, host, got.item())


def test_reduce_ws_back_to_back_and_misaligned(workspace):
    host = host_input("sum_f32", (1 << 22) + 5, seed=2)
    for offset in range(VEC["sum_f32"]):
        x = to_device(host, offset)
        a = abi.rdx_reduce_ws("sum_f32", x, workspace)
        b = abi.rdx_reduce_ws("sum_f32", x, workspace)
        assert torch.equal(as_bits(a), as_bits(b))
        check("sum_f32", host, a.item())


def test_reduce_ws_replays_in_a_cuda_graph(workspace):
    # the workspace variant allocates nothing, so it can be captured and replayed
    n = (1 << 23) + 9
    static_x = torch.empty(n, device=DEV)
    static_out = torch.empty((), device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        static_x.normal_()
        abi.rdx_reduce_ws("sum_f32", static_x, workspace, out=static_out, stream=s)   # warm-up
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        abi.rdx_reduce_ws("sum_f32", static_x, workspace, out=static_out)
    for seed in (11, 12, 13):
        host = inputs.normal_f32(n, seed)
        static_x.copy_(torch.from_numpy(host))
        g.replay()
        torch.cuda.synchronize()
        check("sum_f32", host, static_out.item())


STRIDED = [(3, 5, 5), (3, 5, 6), (7, 3, 8), (33, 255, 257), (100, 256, 300), (64, 1000, 1003), (17, 4099, 4099),
           (5, 5000, 6001), (9, 20000, 20001), (2, 100_000, 130_000), (1000, 64, 67)]


@pytest.mark.parametrize("shape", STRIDED, ids=str)
def test_strided_rowsum_parity(shape):
    rows, cols, ld = shape
    full = inputs.uniform_f32(rows * ld, seed=rows + cols + ld, lo=-1.0, hi=1.0).reshape(rows, ld)
    x = torch.from_numpy(full).to(DEV)[:, :cols]              # a column slice: stride(0) = ld
    got = abi.rdx_rowsum_strided_f32(x).cpu().numpy().astype(np.float64)
    host = np.ascontiguousarray(full[:, :cols])
    ref = oracle.rowsum_f32(host)
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    assert np.all(np.abs(got - ref) <= tol)
    # an offset slice: rows start at column 1 (no row is 16-byte aligned when ld % 4 == 0)
    if cols > 1:
        x1 = torch.from_numpy(full).to(DEV)[:, 1:cols]
        got1 = abi.rdx_rowsum_strided_f32(x1).cpu().numpy().astype(np.float64)
        h1 = np.ascontiguousarray(full[:, 1:cols])
        assert np.all(np.abs(got1 - oracle.rowsum_f32(h1)) <= 1e-6 * oracle.rowabssum_f32(h1) + 1e-30)


SPLIT = [(1, 16384), (1, 100_003), (2, 1 << 20), (3, (1 << 20) + 5), (7, 65536), (64, 20000), (500, 16387),
         (1, 1 << 24), (4, (1 << 22) + 1)]


@pytest.mark.parametrize("shape", SPLIT, ids=str)
def test_split_row_path_parity(shape):
    rows, cols = shape
    host = inputs.normal_f32(rows * cols, seed=rows * 7 + cols % 1000).reshape(rows, cols)
    x = torch.from_numpy(host).to(DEV)
    got = abi.rdx_rowsum_f32(x)
    again = abi.rdx_rowsum_f32(x)
    assert torch.equal(got.view(torch.int32), again.view(torch.int32))
    ref = oracle.rowsum_f32(host)
    tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
    assert np.all(np.abs(got.cpu().numpy().astype(np.float64) - ref) <= tol)


def test_split_rows_with_leading_dimension():
    rows, cols, ld = 5, (1 << 20) + 3, (1 << 20) + 17
    full = inputs.normal_f32(rows * ld, seed=5).reshape(rows, ld)
    x = torch.from_numpy(full).to(DEV)[:, 2:2 + cols]
    host = np.ascontiguousarray(full[:, 2:2 + cols])
    got = abi.rdx_rowsum_strided_f32(x).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - oracle.rowsum_f32(host)) <= 1e-6 * oracle.rowabssum_f32(host) + 1e-30)


@pytest.mark.slow
def test_split_rows_one_gib():
    rows, cols = 4, 1 << 26          # 1 GiB in four rows: each row over many blocks
    x = torch.ones((rows, cols), device=DEV)
    x[1] = -0.5
    x[3, ::2] = 3.0
    got = abi.rdx_rowsum_f32(x).tolist()
    assert got == [float(cols), -0.5 * cols, float(cols), 2.0 * cols]


@pytest.mark.slow
def test_row_offsets_past_2_to_the_32():
    # short rows: 2^25 + 3 rows of 128 columns (more than 2^32 elements, 16 GiB)
    rows = (1 << 25) + 3
    x = torch.ones((rows, 128), device=DEV)
    x[-1] = 2.0
    got = abi.rdx_rowsum_f32(x)
    assert torch.all(got[:-1] == 128.0) and got[-1].item() == 256.0
    del x, got
    torch.cuda.empty_cache()
    # the split path: 2 rows of 2^31 + 7 columns (16 GiB), each over many blocks
    cols = (1 << 31) + 7
    x = torch.ones((2, cols), device=DEV)
    x[1] = -0.25
    got = abi.rdx_rowsum_f32(x).tolist()
    assert abs(got[0] - cols) <= 1e-6 * cols and abs(got[1] + 0.25 * cols) <= 1e-6 * 0.25 * cols
    del x
    torch.cuda.empty_cache()


def test_row_sums_replay_in_a_cuda_graph():
    # the row kernels other than the split path use no workspace, so a capture
    # on the current (capturing) stream with no stream argument replays them
    shapes = [(50_000, 3), (20_000, 12), (20_000, 256), (3000, 2000), (3000, 16384)]
    xs = [torch.empty(shape, device=DEV) for shape in shapes]
    outs = [torch.empty(shape[0], device=DEV) for shape in shapes]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for x, o in zip(xs, outs):
            abi.rdx_rowsum_f32(x.normal_(), out=o)  # warm-up
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, o in zip(xs, outs):
            abi.rdx_rowsum_f32(x, out=o)
    for seed in (21, 22):
        hosts = []
        for k, x in enumerate(xs):
            host = inputs.uniform_f32(x.numel(), seed + k, lo=-1.0, hi=1.0).reshape(x.shape)
            x.copy_(torch.from_numpy(host))
            hosts.append(host)
        g.replay()
        torch.cuda.synchronize()
        for host, o in zip(hosts, outs):
            tol = 1e-6 * oracle.rowabssum_f32(host) + 1e-30
            assert np.all(np.abs(o.cpu().numpy().astype(np.float64) - oracle.rowsum_f32(host)) <= tol)


def test_word_finishing_ops_replay_in_a_cuda_graph(workspace):
    # The int64 sum and the maxima finish through the workspace's accumulator
    # word, which every launch must leave clear: one graph holding all three,
    # replayed on new inputs, gives each op's exact result every time.
    n = (1 << 22) + 3
    xi = torch.empty(n, dtype=torch.int32, device=DEV)
    xf = torch.empty(n, device=DEV)
    outs = [torch.empty((), dtype=torch.int64, device=DEV), torch.empty((), dtype=torch.int32, device=DEV),
            torch.empty((), device=DEV)]
    ops = [("sum_i32", xi), ("max_i32", xi), ("max_f32", xf)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        xi.zero_()
        xf.zero_()
        for (op, x), out in zip(ops, outs):
            abi.rdx_reduce_ws(op, x, workspace, out=out, stream=s)   # warm-up
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (op, x), out in zip(ops, outs):
            abi.rdx_reduce_ws(op, x, workspace, out=out)
    for seed in (21, 22, 23):
        zi = inputs.integers_i32(n, seed, -(2 ** 31), 2 ** 31 - 1)
        zf = inputs.normal_f32(n, seed)
        xi.copy_(torch.from_numpy(zi))
        xf.copy_(torch.from_numpy(zf))
        g.replay()
        torch.cuda.synchronize()
        assert outs[0].item() == oracle.sum_i32(zi)
        assert outs[1].item() == oracle.max_i32(zi)
        assert outs[2].item() == oracle.max_f32(zf)


def test_two_kernel_calls_replay_in_a_cuda_graph(workspace):
    # Inputs of 64 MiB and more finish in a second kernel launched behind the
    # tiles with programmatic dependent launch; a graph of such calls (a
    # partials finish and a word finish, back to back) keeps both kernels
    # and their order, replay after replay.
    n = (1 << 24) + 13
    assert abi.rdx_reduce_kernels("sum_f32", n) == 2 and abi.rdx_reduce_kernels("sum_i32", n) == 2
    xf = torch.empty(n, device=DEV)
    xi = torch.empty(n, dtype=torch.int32, device=DEV)
    of = torch.empty((), device=DEV)
    oi = torch.empty((), dtype=torch.int64, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        xf.zero_()
        xi.zero_()
        abi.rdx_reduce_ws("sum_f32", xf, workspace, out=of, stream=s)   # warm-up
        abi.rdx_reduce_ws("sum_i32", xi, workspace, out=oi, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        abi.rdx_reduce_ws("sum_f32", xf, workspace, out=of)
        abi.rdx_reduce_ws("sum_i32", xi, workspace, out=oi)
    for seed in (31, 32):
        hf = inputs.normal_f32(n, seed)
        hi = inputs.integers_i32(n, seed, -(2 ** 31), 2 ** 31 - 1)
        xf.copy_(torch.from_numpy(hf))
        xi.copy_(torch.from_numpy(hi))
        g.replay()
        torch.cuda.synchronize()
        check("sum_f32", hf, of.item())
        assert oi.item() == oracle.sum_i32(hi)


def test_release_stream_frees_and_the_next_call_reallocates():
    n = (1 << 22) + 5                      # several tiles: the call uses the stream's workspace
    host = host_input("sum_f32", n, seed=41)
    x = to_device(host)
    s = torch.cuda.Stream(DEV)
    first = abi.rdx_sum_f32(x, stream=s)
    s.synchronize()
    assert abi.rdx_release_stream(s) is True
    assert abi.rdx_release_stream(s) is False       # nothing left to free
    again = abi.rdx_sum_f32(x, stream=s)             # a fresh workspace, the same bits
    s.synchronize()
    assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    check("sum_f32", host, again.item())
    assert abi.rdx_release_stream(s) is True
    small = abi.rdx_sum_f32(x[:1000], stream=s)      # one tile: no workspace needed
    s.synchronize()
    assert abi.rdx_release_stream(s) is False
    check("sum_f32", host[:1000], small.item())
