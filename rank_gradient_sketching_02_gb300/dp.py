"""Data-parallel exchange of the sketch.

The sketch is linear in the gradient and A is a pure function of (seed, step),
so data-parallel ranks that each accumulate their own microbatches only need
one sum-all-reduce of S (d x r) per matrix before the apply; no projection
matrix is communicated.  That all-reduce is k/r times smaller than the
gradient's (theclarity.today write-up, "Why it matters": nodes exchange the
compact sketch).
"""
from __future__ import annotations


def allreduce_sketch(S, group=None):
    """Sum S over the ranks of ``group`` in place (torch.distributed, any backend)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(S, op=dist.ReduceOp.SUM, group=group)
    return S


def shard_microbatches(n_microbatches: int, rank: int, world: int):
    """Microbatch indices of ``rank`` when a step's microbatches are split over ``world`` ranks."""
    return list(range(rank, n_microbatches, world))
