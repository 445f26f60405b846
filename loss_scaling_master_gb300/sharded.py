"""Data-parallel sharding of the optimizer step (ZeRO-style ownership).

Every element of the step is independent except the non-finite flag: each
rank checks only the gradients it owns, and all ranks must skip together, so
the one exchange is an all-reduce(MAX) of the int32 ``found_inf`` between the
check and the update ("第20章 量化与混合精度训练" §20.5.33: per-device flags are
combined before the scale update).  With gradient-norm clipping the global
norm is the square root of the sum of the ranks' sums of squares, a second
all-reduce (SUM) of one fp64 value.  Whole tensors are owned by one rank, so
the per-tensor FP8 amax needs no exchange.
"""
from __future__ import annotations


def partition_tensors(numels, world: int):
    """Assign whole tensors to ranks, largest first to the least-loaded rank.
    Returns one list of tensor indices per rank (each sorted)."""
    load = [0] * world
    owned = [[] for _ in range(world)]
    for i in sorted(range(len(numels)), key=lambda i: (-numels[i], i)):
        r = min(range(world), key=lambda r: (load[r], r))
        owned[r].append(i)
        load[r] += numels[i]
    return [sorted(o) for o in owned]


def combine_found_inf(found_inf, group=None):
    """In-place all-reduce(MAX) of the int32 flag tensor across the group."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(found_inf, op=dist.ReduceOp.MAX, group=group)
    return found_inf


def combine_grad_sumsq(grad_sumsq, group=None):
    """In-place all-reduce(SUM) of the fp64 sum of squared unscaled gradients."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(grad_sumsq, op=dist.ReduceOp.SUM, group=group)
    return grad_sumsq
