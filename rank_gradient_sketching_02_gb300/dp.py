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


class SketchArena:
    """The sketches of many matrices as views of one contiguous fp32 buffer.

    A data-parallel step exchanges one S per compressed matrix (196 for a
    28-layer model with seven projections per layer).  Held as views of one
    buffer, they are zeroed at the start of a step by one fill and summed over
    the ranks by one all-reduce per bucket: consecutive views packed up to
    ``bucket_bytes`` (a view larger than that is a bucket of its own), so the
    collective count no longer grows with the matrix count and no S is copied
    into or out of a staging buffer.  Every view starts on a 16-byte boundary
    (d * r is a multiple of 32 floats), as the library's sketch calls require.

    Buckets follow the order of ``shapes``; ``bucket_of(i)`` gives the bucket
    that holds matrix i, so a caller can reduce a bucket as soon as its last
    matrix's final microbatch has been sketched (the backward pass finishes the
    last layers first) while later sketches still run.
    """

    def __init__(self, shapes, r: int, device=None, bucket_bytes: int = 64 << 20):
        import torch
        if r <= 0 or r % 32:
            raise ValueError(f"rank {r} is not a positive multiple of 32")
        self.r = int(r)
        self.shapes = [int(d) for d in shapes]
        if any(d <= 0 for d in self.shapes):
            raise ValueError("every sketch needs d >= 1 rows")
        offs, total = [], 0
        for d in self.shapes:
            offs.append(total)
            total += d * self.r
        self.flat = torch.zeros(total, dtype=torch.float32, device=device)
        self.S = [self.flat[o:o + d * self.r].view(d, self.r) for o, d in zip(offs, self.shapes)]
        cap = max(1, int(bucket_bytes) // 4)
        self.buckets = []            # (first element, end element, first matrix, end matrix)
        self._bucket_of = []
        start, first = 0, 0
        for i, (o, d) in enumerate(zip(offs, self.shapes)):
            end = o + d * self.r
            if end - start > cap and i > first:
                self.buckets.append((start, o, first, i))
                start, first = o, i
            self._bucket_of.append(len(self.buckets))
        if self.shapes:
            self.buckets.append((start, total, first, len(self.shapes)))

    def __len__(self):
        return len(self.S)

    def __getitem__(self, i):
        return self.S[i]

    def bucket_of(self, i: int) -> int:
        """Index of the bucket holding matrix i."""
        return self._bucket_of[i]

    def zero_(self):
        """Zero every sketch (the first microbatch of a step adds into zeros)."""
        self.flat.zero_()
        return self

    def allreduce_bucket(self, b: int, group=None):
        """Sum bucket ``b`` over the ranks of ``group`` in place (see allreduce_sketch)."""
        s, e, _, _ = self.buckets[b]
        allreduce_sketch(self.flat[s:e], group)

    def allreduce(self, group=None):
        """Sum every sketch over the ranks of ``group``, one collective per bucket."""
        for b in range(len(self.buckets)):
            self.allreduce_bucket(b, group)
        return self
