"""Data-parallel sharding of the optimizer step.

Two ownership layouts:

* whole tensors (``partition_tensors``, ZeRO-style): every tensor belongs to
  one rank.  Every element of the step is independent except the non-finite
  flag: each rank checks only the gradients it owns and all ranks must skip
  together, so the one exchange is an all-reduce(MAX) of the int32
  ``found_inf`` between the check and the update ("第20章 量化与混合精度训练"
  §20.5.33: per-device flags are combined before the scale update).  With
  gradient-norm clipping the global norm is the square root of the sum of
  the ranks' sums of squares, a second all-reduce (SUM) of one fp64 value.

* flat shards (``partition_flat``, FSDP-style: §20.5.26 "AMP × FSDP" shards
  flat parameters): the tensors laid end to end as one flat parameter, cut
  into one contiguous slice per rank, so a tensor can span ranks.  A 2-D
  weight with an FP8 copy is then cut between whole rows: its piece on a
  rank is a band of rows, whose FP8 bytes are those rows of the FP8 copy and
  whose transposed bytes are the matching column slice of the transposed
  copy.  The per-tensor amax of such a weight is a max over every rank's
  piece, so it is all-reduced (MAX) between the update, which folds each
  piece's max|bf16|, and the FP8 cast (``combine_amax``).

The collectives run on the caller's process group; NCCL on GPUs, gloo on
CPU.  The pages describe no wire format of their own.
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


def partition_flat(shapes, world: int, row_align: int = 16, elem_align: int = 8):
    """Cut the flat parameter (the tensors of ``shapes`` end to end, in order)
    into ``world`` contiguous slices of about equal size.

    shapes: per tensor (n,) for a 1-D tensor or (rows, cols) for a 2-D one.
    Each of the world - 1 cuts starts at r * N / world (N the total size) and
    moves to the nearest multiple of ``row_align`` whole rows of the 2-D
    tensor it falls in (so 2-D pieces are bands of whole rows, 16-byte
    aligned in both FP8 layouts when row_align is 16), or of ``elem_align``
    elements of a 1-D tensor (16-byte aligned views of 16-bit data), never
    past either end of that tensor.  Returns, per rank, the pieces
    (tensor index, begin, end) in elements of the tensor, in flat order;
    a rank's slice may be empty."""
    sizes = [int(s[0]) * (int(s[1]) if len(s) > 1 else 1) for s in shapes]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += n
    cuts = [0]
    for r in range(1, world):
        target = (r * total) // world
        t = 0
        while t + 1 < len(sizes) and offs[t + 1] <= target:
            t += 1
        if not sizes:
            cuts.append(0)
            continue
        unit = row_align * int(shapes[t][1]) if len(shapes[t]) > 1 else elem_align
        p = target - offs[t]
        p = min(sizes[t], max(0, int(round(p / unit)) * unit))
        cuts.append(max(cuts[-1], offs[t] + p))
    cuts.append(total)
    out = []
    for r in range(world):
        lo, hi, pieces = cuts[r], cuts[r + 1], []
        for t, (o, n) in enumerate(zip(offs, sizes)):
            b, e = max(lo, o), min(hi, o + n)
            if e > b:
                pieces.append((t, b - o, e - o))
        out.append(pieces)
    return out


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


def combine_amax(amax, group=None):
    """In-place all-reduce(MAX) of the per-tensor fp32 amax array.  The values
    are magnitudes (or NaN), whose fp32 bit patterns order like the values with
    NaN above infinity, so the reduction runs on the int32 view: a NaN on any
    rank stays NaN, which a float max would not promise."""
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax.view(torch.int32), op=dist.ReduceOp.MAX, group=group)
    return amax
