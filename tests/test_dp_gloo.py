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
