"""Reductions split over several GPUs: one process per GPU, torch.distributed.

The page "03_shared_memory_sync_reduction.py", demo 3, reduces in two stages:
every block leaves one partial, and a second step outside the kernel adds the
partials (demo 2 of the page: blocks exchange data only by ending the
kernel).  Split over P GPUs the same two stages appear one level up:

1. rank r takes its chunk of the array (``rdx_shard_range``: contiguous,
   balanced, chunk starts 16-byte aligned relative to the array) and reduces
   it with the one-GPU entry point, leaving one partial on its device;
2. the partials are all-gathered in rank order (the one exchange: a
   torch.distributed collective, NCCL between GPUs);
3. every rank adds the P partials in rank order (``rdx_combine_*``), so every
   rank holds the same bits, run after run.

Row sums split by rows (granule 1) and need no exchange: rank r's rows give
its slice of the output.

``emulate`` runs the same split on one GPU: the chunks one after another into
the slots of one partials array, then the combine.  Each chunk is its own
launch and nothing waits on anything but stream order, so it is the same set
of additions that P GPUs make, in the same order: for an array whose base is
16-byte aligned (every chunk then starts 16-byte aligned, as a chunk in a
fresh allocation does) the result has the same bits.

This module only chooses chunks and moves partials; every addition happens
in the library's kernels.
"""
from __future__ import annotations

import torch

from . import abi

# Elements per granule: 16 bytes of the element type (chunk starts keep the
# whole array's 16-byte alignment), one row for row sums.
GRANULE = {"sum_f32": 4, "sumsq_f32": 4, "sum_i32": 4, "sum_bf16": 8, "sumsq_bf16": 8,
           "sum_sumsq_f32": 4, "sum_sumsq_bf16": 8, "rowsum_f32": 1}

_ENTRY = {"sum_f32": abi.rdx_sum_f32, "sumsq_f32": abi.rdx_sumsq_f32, "sum_i32": abi.rdx_sum_i32_i64,
          "sum_bf16": abi.rdx_sum_bf16_f32acc, "sumsq_bf16": abi.rdx_sumsq_bf16_f32acc,
          "sum_sumsq_f32": abi.rdx_sum_sumsq_f32, "sum_sumsq_bf16": abi.rdx_sum_sumsq_bf16_f32acc}

# (combine entry point, partial dtype, partial shape)
_COMBINE = {"sum_f32": (abi.rdx_combine_f32, torch.float32, ()),
            "sumsq_f32": (abi.rdx_combine_f32, torch.float32, ()),
            "sum_bf16": (abi.rdx_combine_f32, torch.float32, ()),
            "sumsq_bf16": (abi.rdx_combine_f32, torch.float32, ()),
            "sum_i32": (abi.rdx_combine_i64, torch.int64, ()),
            "sum_sumsq_f32": (abi.rdx_combine_f32x2, torch.float32, (2,)),
            "sum_sumsq_bf16": (abi.rdx_combine_f32x2, torch.float32, (2,))}

OPS = tuple(_ENTRY)


def shard_range(op: str, n: int, world: int, rank: int) -> tuple[int, int]:
    """[lo, hi): rank ``rank``'s chunk of ``n`` elements (rows for
    ``rowsum_f32``) among ``world`` ranks."""
    return abi.rdx_shard_range(n, world, rank, GRANULE[op])


def local_chunk(op: str, x: torch.Tensor, world: int, rank: int) -> torch.Tensor:
    """Rank ``rank``'s chunk of ``x``: a flat slice for the scalar
    reductions, a slice of rows for ``rowsum_f32``."""
    if op == "rowsum_f32":
        lo, hi = shard_range(op, x.shape[0], world, rank)
        return x[lo:hi]
    lo, hi = shard_range(op, x.numel(), world, rank)
    return x.reshape(-1)[lo:hi]


def local_partial(op: str, x_local: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """This rank's partial: the one-GPU reduction ``op`` of its chunk."""
    return _ENTRY[op](x_local, out=out, stream=stream)


def combine(op: str, parts: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The gathered partials of ``op`` (rank order along dim 0) added in rank
    order on the device (rdx_combine_f32, _f32x2 or _i64)."""
    return _COMBINE[op][0](parts, out=out, stream=stream)


def partial_spec(op: str):
    """(dtype, shape) of one partial of ``op``."""
    _, dtype, shape = _COMBINE[op]
    return dtype, shape


def gather_partials(partial: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's ``partial`` stacked in rank order: a (world, *shape)
    tensor on ``partial``'s device, identical on every rank."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    partial = partial.contiguous()
    out = torch.empty((world, *partial.shape), dtype=partial.dtype, device=partial.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(out, partial, group=group)
    else:
        dist.all_gather(list(out.unbind(0)), partial, group=group)
    return out


def sharded_reduce(op: str, x_local: torch.Tensor, group=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """The reduction ``op`` of the whole array from this rank's chunk of it
    (``local_chunk``): the chunk's partial, an all-gather of the partials,
    and their sum in rank order.  Runs on the current CUDA stream; every
    rank returns the same bits."""
    return combine(op, gather_partials(local_partial(op, x_local), group), out=out)


def sharded_rowsum(x_local_rows: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Row sums of this rank's rows (``local_chunk("rowsum_f32", ...)``): the
    rank's slice of the whole output.  Rows do not span ranks, so there is
    nothing to exchange."""
    return abi.rdx_rowsum_f32(x_local_rows, out=out)


def emulate(op: str, x: torch.Tensor, parts: int, out: torch.Tensor | None = None,
            partials: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The split of ``sharded_reduce`` over ``parts`` ranks, run on one GPU:
    chunk r's partial into slot r of ``partials`` (allocated if None), then
    the combine in rank order.  ``x`` is the whole array."""
    dtype, shape = partial_spec(op)
    flat = x.reshape(-1)
    if partials is None:
        partials = torch.empty((parts, *shape), dtype=dtype, device=x.device)
    for r in range(parts):
        lo, hi = shard_range(op, flat.numel(), parts, r)
        local_partial(op, flat[lo:hi], out=partials[r], stream=stream)
    return combine(op, partials, out=out, stream=stream)
