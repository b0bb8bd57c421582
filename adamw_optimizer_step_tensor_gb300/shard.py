"""Data-parallel sharding of the optimizer step (host-side logic).

The AdamW update is elementwise, so N ranks can each own a disjoint contiguous
slice of the flattened parameter space (optimizer-state sharding, as the
DTensor/FSDP ``Shard(0)`` discussion on "Adam-mini <> DTensor" does for whole
parameters) and step it with their own plan, with no exchange inside the step.
The one thing the ranks must agree on is whether to skip: each rank checks its
own grads and the flags are combined with an all-reduce MAX before the step
("FusedAdam & PyTorch Lightning AMP": one non-finite grad anywhere skips the
whole step).

Tensors are laid out in the flattened space at offsets rounded up to ``align``
elements (256 by default: one 8-bit state block), and shard boundaries are
multiples of ``align``, so a shard never splits an 8-bit block of a tensor.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Slice:
    tensor: int   # index into the tensor list
    start: int    # first element inside that tensor
    stop: int     # one past the last element


def padded_offsets(numels: list[int], align: int = 256) -> tuple[list[int], int]:
    """Flattened start of every tensor (multiples of ``align``) and the padded total."""
    offs, o = [], 0
    for n in numels:
        offs.append(o)
        o += (n + align - 1) // align * align
    return offs, o


def shard_bounds(total: int, world: int, rank: int, align: int = 256) -> tuple[int, int]:
    """[lo, hi) of rank's share of ``total`` padded elements, in whole ``align`` units."""
    if not (0 <= rank < world):
        raise ValueError("rank out of range")
    units = (total + align - 1) // align
    per, extra = divmod(units, world)
    lo = rank * per + min(rank, extra)
    hi = lo + per + (1 if rank < extra else 0)
    return min(lo * align, total), min(hi * align, total)


def shard_slices(numels: list[int], world: int, rank: int, align: int = 256) -> list[Slice]:
    """The pieces of each tensor that rank owns (empty pieces omitted)."""
    offs, total = padded_offsets(numels, align)
    lo, hi = shard_bounds(total, world, rank, align)
    out = []
    for i, (o, n) in enumerate(zip(offs, numels)):
        a, b = max(lo, o), min(hi, o + n)
        if a < b:
            out.append(Slice(i, a - o, b - o))
    return out


def allreduce_found_inf(found_inf, group=None) -> None:
    """Combine every rank's found-inf flag (a float32 tensor of one element) in place: MAX."""
    import torch.distributed as dist
    dist.all_reduce(found_inf, op=dist.ReduceOp.MAX, group=group)
