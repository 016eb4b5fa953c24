"""Data-parallel sketch exchange on CPU ranks (gloo, world size 2).

The sketch is linear in the gradient and A depends only on (seed, step), so
ranks that sketch disjoint microbatches and sum-all-reduce S hold exactly the
single-process sketch of all microbatches.  A rank that drops out before the
exchange is detected by the survivor as an error, not a hang.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import logra_oracle as O

D, K, R, N, MBS = 24, 136, 32, 40, 6


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _microbatches():
    g = np.random.default_rng(5)
    return [(g.standard_normal((N, K)), g.standard_normal((N, D))) for _ in range(MBS)]


def _init(rank, world, port, timeout_s=30):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _worker_sum(rank, world, port, out):
    from rank_gradient_sketching_02_gb300 import dp
    _init(rank, world, port)
    S = np.zeros((D, R))
    for i in dp.shard_microbatches(MBS, rank, world):
        X, dY = _microbatches()[i]
        S = O.sketch_accumulate(S, X, dY, 11, 3, R)
    t = torch.from_numpy(S)
    dp.allreduce_sketch(t)
    np.save(os.path.join(out, f"S{rank}.npy"), t.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_allreduced_shards_equal_single_rank_sketch(tmp_path):
    port = _free_port()
    mp.start_processes(_worker_sum, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    S_single = np.zeros((D, R))
    for X, dY in _microbatches():
        S_single = O.sketch_accumulate(S_single, X, dY, 11, 3, R)
    for rank in range(2):
        S = np.load(tmp_path / f"S{rank}.npy")
        np.testing.assert_allclose(S, S_single, rtol=1e-12, atol=1e-12)


def _worker_drop(rank, world, port, out):
    from rank_gradient_sketching_02_gb300 import dp
    _init(rank, world, port, timeout_s=5)
    if rank == 1:
        os._exit(0)            # leaves between steps, before the exchange
    t = torch.ones((D, R), dtype=torch.float64)
    try:
        dp.allreduce_sketch(t)
        result = "no-error"
    except Exception as e:  # noqa: BLE001 - any distributed error is the detection
        result = "error:" + type(e).__name__
    with open(os.path.join(out, "drop.txt"), "w") as f:
        f.write(result)
    os._exit(0)


def test_dropped_rank_is_detected(tmp_path):
    port = _free_port()
    ctx = mp.start_processes(_worker_drop, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn",
                             join=False)
    import time
    deadline = time.time() + 90
    while time.time() < deadline and any(p.is_alive() for p in ctx.processes):
        time.sleep(0.5)
    for p in ctx.processes:
        if p.is_alive():
            p.kill()
    res = (tmp_path / "drop.txt").read_text()
    assert res.startswith("error:"), res


def test_shard_microbatches_partition():
    from rank_gradient_sketching_02_gb300 import dp
    for world in (1, 2, 3, 8):
        got = sorted(i for r in range(world) for i in dp.shard_microbatches(16, r, world))
        assert got == list(range(16))


ARENA_D = (24, 8, 64, 8, 8, 96)    # several matrices of one rank r, packed into one buffer


def _worker_arena(rank, world, port, out):
    from rank_gradient_sketching_02_gb300 import dp
    _init(rank, world, port)
    # buckets of at most two 24 x 32 sketches' worth of bytes: 24 + 8 rows share one, the 64-row
    # sketch is one of its own, 8 + 8 rows share one and the 96-row sketch (larger than a bucket)
    # is one of its own: four collectives
    arena = dp.SketchArena(ARENA_D, R, bucket_bytes=2 * 24 * R * 4)
    arena.flat.fill_(7.0)
    arena.zero_()                  # the first microbatch of a step adds into zeros
    for m, d in enumerate(ARENA_D):
        S = np.zeros((d, R))
        for i in dp.shard_microbatches(MBS, rank, world):
            X, dY = _microbatches()[i]
            S = O.sketch_accumulate(S, X, dY[:, :1].repeat(d, axis=1) * (m + 1), 20 + m, 3, R)
        arena[m].copy_(torch.from_numpy(S).float())
    arena.allreduce()
    np.save(os.path.join(out, f"A{rank}.npy"), arena.flat.numpy())
    np.save(os.path.join(out, f"buckets{rank}.npy"), np.array(arena.buckets))
    dist.barrier()
    dist.destroy_process_group()


def test_arena_exchange_in_buckets_equals_single_rank_sketches(tmp_path):
    port = _free_port()
    mp.start_processes(_worker_arena, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    want = []
    for m, d in enumerate(ARENA_D):
        S = np.zeros((d, R))
        for X, dY in _microbatches():
            S = O.sketch_accumulate(S, X, dY[:, :1].repeat(d, axis=1) * (m + 1), 20 + m, 3, R)
        want.append(S.astype(np.float32).astype(np.float64).ravel())
    want = np.concatenate(want)
    buckets = np.load(tmp_path / "buckets0.npy")
    assert [tuple(b[2:]) for b in buckets] == [(0, 2), (2, 3), (3, 5), (5, 6)] and buckets[-1][1] == want.size
    for rank in range(2):
        got = np.load(tmp_path / f"A{rank}.npy").astype(np.float64)
        # each rank's shard was rounded to fp32 before the sum: fp32-sized differences only
        np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6 * np.abs(want).max())


def test_arena_views_layout():
    from rank_gradient_sketching_02_gb300 import dp
    a = dp.SketchArena((3584, 512, 18944), 256, bucket_bytes=16 << 20)
    assert [tuple(s.shape) for s in a.S] == [(3584, 256), (512, 256), (18944, 256)]
    assert all(s.data_ptr() % 16 == 0 and s.is_contiguous() for s in a.S)
    assert a.S[1].data_ptr() == a.S[0].data_ptr() + 3584 * 256 * 4          # views of one buffer
    a.S[2].fill_(1.0)
    assert float(a.flat.sum()) == 18944 * 256
    a.zero_()
    assert float(a.flat.abs().sum()) == 0.0
    # 3.7 MB + 0.5 MB share a bucket; the 19.4 MB sketch is a bucket of its own
    assert [b[2:] for b in a.buckets] == [(0, 2), (2, 3)]
    assert [a.bucket_of(i) for i in range(3)] == [0, 0, 1]
    with pytest.raises(ValueError):
        dp.SketchArena((8,), 48)
