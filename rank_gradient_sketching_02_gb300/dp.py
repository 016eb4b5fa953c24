"""Data-parallel exchange of the sketch.

The sketch is linear in the gradient and A is a pure function of (seed, step),
so data-parallel ranks that each accumulate their own microbatches only need
one sum-all-reduce of S (d x r) per matrix before the apply; no projection
matrix is communicated.  That all-reduce is k/r times smaller than the
gradient's (theclarity.today write-up, "Why it matters": nodes exchange the
compact sketch).  After it every rank holds the same S bits, and the apply is
deterministic for given S bits, so ranks that each apply RowAdam keep
bit-identical weights without exchanging them.
"""
from __future__ import annotations


def _host_only_backend(group) -> bool:
    """True when the group's backend reduces host tensors only (gloo)."""
    import torch.distributed as dist
    return str(dist.get_backend(group)).lower() == "gloo"


def allreduce_sketch(S, group=None):
    """Sum S over the ranks of ``group`` in place (torch.distributed, any backend).

    With NCCL the device tensor is reduced where it lies.  With a host-only
    backend (gloo, e.g. ranks without NCCL or CPU-side test ranks) a device S
    is staged through host memory: copied out, reduced, copied back, on the
    current stream, so the call stays ordered with the sketch calls before it
    and the apply after it.
    """
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) <= 1:
        return S
    if S.is_cuda and _host_only_backend(group):
        host = S.detach().to("cpu")            # waits for the sketches that produced S
        dist.all_reduce(host, op=dist.ReduceOp.SUM, group=group)
        S.copy_(host)
        return S
    dist.all_reduce(S, op=dist.ReduceOp.SUM, group=group)
    return S


def shard_microbatches(n_microbatches: int, rank: int, world: int):
    """Microbatch indices of ``rank`` when a step's microbatches are split over ``world`` ranks."""
    return list(range(rank, n_microbatches, world))
