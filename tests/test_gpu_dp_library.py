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
