"""Two data-parallel ranks running the CUDA library, exchanging S over gloo.

Each rank is its own process on the same GPU (their kernels never wait on one
another), sketches a disjoint share of a step's microbatches through the C
ABI, and sums its S with the other rank's through `dp.allreduce_sketch`
(gloo, staged through host memory).  Both ranks must then hold the oracle
sketch of all microbatches (1e-3, bf16 inputs) and identical S bits, and a
RowAdam apply on each rank must give bit-identical weights (the apply is
deterministic for given S bits).  The NCCL path is the same call on device
tensors; it is not run here (one GPU).
"""
import datetime
import os
import socket

import numpy as np
import pytest

from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

N, D, K, R, MBS, SEED, STEP = 1000, 1032, 1544, 256, 6, 4242, 9


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _mb(i):
    X, dY, _ = synth.host_microbatch(N, D, K, dy_kind="lognormal", mask_frac=0.25, key=(31, i))
    return synth.to_bf16_bits(X), synth.to_bf16_bits(dY)


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(0)
    import rank_gradient_sketching_02_gb300 as L
    from rank_gradient_sketching_02_gb300 import dp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    S = torch.zeros((D, R), dtype=torch.float32, device="cuda")
    for i in dp.shard_microbatches(MBS, rank, world):
        X, dY = _mb(i)
        L.logra_sketch_accumulate(X.cuda(), dY.cuda(), S, SEED, STEP)
    dp.allreduce_sketch(S)
    W = torch.zeros((D, K), dtype=torch.float32, device="cuda")
    v = torch.zeros(D, dtype=torch.float32, device="cuda")
    L.logra_rowadam_apply(W, S, v, SEED, STEP, 0.999, 1e-8, 1e-5, 1.0)
    torch.cuda.synchronize()
    status = L.logra_get_status()
    np.save(os.path.join(out, f"S{rank}.npy"), S.cpu().numpy())
    np.save(os.path.join(out, f"W{rank}.npy"), W.cpu().numpy())
    with open(os.path.join(out, f"status{rank}.txt"), "w") as f:
        f.write(str(status))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_allreduce_library_sketches(tmp_path):
    import torch.multiprocessing as mp
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    mp.start_processes(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    S_or = np.zeros((D, R))
    for i in range(MBS):
        X, dY = _mb(i)
        S_or = O.sketch_accumulate(S_or, X.double().numpy(), dY.double().numpy(), SEED, STEP, R)
    S0, S1 = np.load(tmp_path / "S0.npy"), np.load(tmp_path / "S1.npy")
    for rank in range(2):
        assert (tmp_path / f"status{rank}.txt").read_text() == "0"
    assert np.array_equal(S0.view(np.uint32), S1.view(np.uint32))
    err = np.linalg.norm(S0.astype(np.float64) - S_or) / np.linalg.norm(S_or)
    assert err <= 1e-3, err
    W0, W1 = np.load(tmp_path / "W0.npy"), np.load(tmp_path / "W1.npy")
    assert np.array_equal(W0.view(np.uint32), W1.view(np.uint32))
    assert np.any(W0)


def test_arena_views_are_library_sketches():
    """The sketches of several matrices as views of one dp.SketchArena buffer: each view is a
    16-byte-aligned d x r tensor the library adds into like any other S, a fill zeroes them all,
    and a grouped apply reads them in place.  Views must not bleed into their neighbours."""
    import torch
    from rank_gradient_sketching_02_gb300 import build as B
    from rank_gradient_sketching_02_gb300 import dp
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    shapes = [(264, 520), (72, 1032), (1032, 264)]              # (d, k) of three matrices
    arena = dp.SketchArena([d for d, _ in shapes], R, device="cuda")
    arena.flat.fill_(3.0)
    arena.zero_()
    n, want = 300, []
    for m, (d, k) in enumerate(shapes):
        S_or = np.zeros((d, R))
        for mb in range(2):
            X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(32, m, mb))
            Xd, dYd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda()
            L.logra_sketch_accumulate(Xd, dYd, arena[m], 70 + m, STEP)
            S_or = O.sketch_accumulate(S_or, Xd.double().cpu().numpy(), dYd.double().cpu().numpy(), 70 + m, STEP, R)
        want.append(S_or)
    Ws = [torch.zeros((d, k), device="cuda") for d, k in shapes]
    vs = [torch.zeros(d, device="cuda") for d, _ in shapes]
    items = [{"W": Ws[m], "S": arena[m], "v": vs[m], "seed": 70 + m, "lr": 1e-5, "c": 1.0}
             for m in range(len(shapes))]
    L.logra_rowadam_apply_group(items, STEP, 0.999, 1e-8)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    b2, eps, lr = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-5))
    for m, (d, k) in enumerate(shapes):
        S = arena[m].double().cpu().numpy()
        assert np.linalg.norm(S - want[m]) / np.linalg.norm(want[m]) <= 1e-3, m
        _, _, _, dW_or = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 70 + m, STEP, b2, eps, lr, 1.0)
        W = Ws[m].double().cpu().numpy()
        assert np.linalg.norm(W - dW_or) / np.linalg.norm(dW_or) <= 1e-5, m


ARENA_SHAPES = [(264, 520), (1032, 264), (72, 1032)]      # (d, k) of three matrices


def _arena_mb(m, i):
    d, k = ARENA_SHAPES[m]
    X, dY, _ = synth.host_microbatch(300, d, k, dy_kind="lognormal", mask_frac=0.25, key=(33, m, i))
    return synth.to_bf16_bits(X), synth.to_bf16_bits(dY)


def _arena_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(0)
    import rank_gradient_sketching_02_gb300 as L
    from rank_gradient_sketching_02_gb300 import dp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    # buckets of at most the first sketch's bytes: three collectives, one per sketch
    arena = dp.SketchArena([d for d, _ in ARENA_SHAPES], R, device="cuda", bucket_bytes=264 * R * 4)
    arena.zero_()
    for m in range(len(ARENA_SHAPES)):
        for i in dp.shard_microbatches(4, rank, world):
            X, dY = _arena_mb(m, i)
            L.logra_sketch_accumulate(X.cuda(), dY.cuda(), arena[m], SEED + m, STEP)
    arena.allreduce()
    torch.cuda.synchronize()
    np.save(os.path.join(out, f"A{rank}.npy"), arena.flat.cpu().numpy())
    with open(os.path.join(out, f"astatus{rank}.txt"), "w") as f:
        f.write(f"{L.logra_get_status()} {len(arena.buckets)}")
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_exchange_a_sketch_arena_in_buckets(tmp_path):
    """Both ranks run the library into views of one dp.SketchArena and exchange it bucket by
    bucket over gloo: the same bits on both ranks, each sketch within 1e-3 of the oracle sketch of
    all four microbatches."""
    import torch.multiprocessing as mp
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    mp.start_processes(_arena_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    for rank in range(2):
        assert (tmp_path / f"astatus{rank}.txt").read_text() == "0 3"
    A0, A1 = np.load(tmp_path / "A0.npy"), np.load(tmp_path / "A1.npy")
    assert np.array_equal(A0.view(np.uint32), A1.view(np.uint32))
    off = 0
    for m, (d, k) in enumerate(ARENA_SHAPES):
        want = np.zeros((d, R))
        for i in range(4):
            X, dY = _arena_mb(m, i)
            want = O.sketch_accumulate(want, X.double().numpy(), dY.double().numpy(), SEED + m, STEP, R)
        got = A0[off:off + d * R].reshape(d, R).astype(np.float64)
        off += d * R
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-3, m
