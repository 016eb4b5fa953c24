"""logra_sketch_accumulate_group: several sketches from one caller stream, spread by the library over
its own side streams and joined back, against the fp64 oracle.

Items of different shapes, two microbatches sharing one S, results read by ordinary stream-ordered
work right after the call (the join), and the call captured into a CUDA graph and replayed after an
eager apply on the same stream.  S sits between guard regions (tests/canary.py).
"""
import numpy as np
import pytest

from canary import Guarded
from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import torch
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    torch.cuda.init()
    return L


def rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(np.asarray(a, np.float64) - np.asarray(b, np.float64)) / (nb if nb > 0 else 1.0)


def _case(n, shapes, key):
    """shapes: list of (d, k, microbatches); returns host inputs per matrix."""
    mats = []
    for mi, (d, k, nmb) in enumerate(shapes):
        mbs = []
        for mb in range(nmb):
            X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(key, mi, mb))
            mbs.append((synth.to_bf16_bits(X), synth.to_bf16_bits(dY)))
        mats.append((d, k, mbs))
    return mats


@pytest.mark.parametrize("n,r", [(1000, 128), (777, 256), (2048, 512)])
def test_group_matches_oracle_and_orders_later_work(L, n, r):
    import torch
    shapes = [(264, 1032, 2), (1032, 520, 1), (72, 2056, 2), (512, 264, 1)]
    mats = _case(n, shapes, 300 + r)
    step = 6
    S = [Guarded((d, r), torch.float32, fill=0.0) for d, _, _ in mats]
    items = []
    for mi, (d, k, mbs) in enumerate(mats):
        for X, dY in mbs:
            items.append({"X": X.cuda(), "dY": dY.cuda(), "S": S[mi].t, "seed": 1000 + mi})
    L.logra_sketch_accumulate_group(items, step)
    copies = [g.t.clone() for g in S]            # ordinary work on the caller stream, after the join
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    for mi, (d, k, mbs) in enumerate(mats):
        S[mi].check(f"S of matrix {mi}")
        want = np.zeros((d, r))
        for X, dY in mbs:
            want = O.sketch_accumulate(want, X.double().numpy(), dY.double().numpy(), 1000 + mi, step, r)
        assert rel(copies[mi].cpu().numpy(), want) <= 1e-3, mi


def test_group_captured_in_a_graph(L):
    import torch
    n, r, step = 1024, 256, 3
    mats = _case(n, [(264, 1032, 2), (520, 776, 1)], 77)
    dev = [(d, k, [(X.cuda(), dY.cuda()) for X, dY in mbs]) for d, k, mbs in mats]
    S = [torch.zeros((d, r), device="cuda") for d, _, _ in mats]
    items = [{"X": X, "dY": dY, "S": S[mi], "seed": 50 + mi} for mi, (_, _, mbs) in enumerate(dev) for X, dY in mbs]
    s = torch.cuda.Stream()
    W = torch.zeros((512, 776), device="cuda")
    Sa = torch.randn((512, r), device="cuda") * 1e-3
    va = torch.zeros(512, device="cuda")
    with torch.cuda.stream(s):
        L.logra_sketch_accumulate_group(items, step)            # creates the side streams and workspaces
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for t in S:
                t.zero_()
            L.logra_sketch_accumulate_group(items, step)
        for rep in range(2):
            L.logra_rowadam_apply(W, Sa, va, 5, rep, 0.999, 1e-8, 1e-5, 1.0)
            for t in S:
                t.fill_(3.0)
            g.replay()
            torch.cuda.synchronize()
            for mi, (d, k, mbs) in enumerate(mats):
                want = np.zeros((d, r))
                for X, dY in mbs:
                    want = O.sketch_accumulate(want, X.double().numpy(), dY.double().numpy(), 50 + mi, step, r)
                assert rel(S[mi].cpu().numpy(), want) <= 1e-3, (rep, mi)
    assert L.logra_get_status() == 0


def test_group_rejects_mixed_token_counts(L):
    import torch
    a = {"X": torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda"),
         "dY": torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda"),
         "S": torch.zeros((64, 32), device="cuda"), "seed": 1}
    b = dict(a, X=torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda"),
             dY=torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        L.logra_sketch_accumulate_group([a, b], 0)


def test_group_wider_than_the_side_streams(L):
    """More items than the library has side streams (16): items wrap around onto streams already in
    use, and microbatches of one matrix land on different streams and add into one S at once."""
    import torch
    n, r, step = 512, 128, 2
    shapes = [(72 + 8 * (mi % 5), 264 + 64 * (mi % 3), 2) for mi in range(11)]     # 11 matrices, 22 items
    mats = _case(n, shapes, 91)
    S = [Guarded((d, r), torch.float32, fill=0.0) for d, _, _ in mats]
    items = [{"X": X.cuda(), "dY": dY.cuda(), "S": S[mi].t, "seed": 700 + mi}
             for mi, (_, _, mbs) in enumerate(mats) for X, dY in mbs]
    assert len(items) > 16
    L.logra_sketch_accumulate_group(items, step)
    copies = [g.t.clone() for g in S]            # ordinary work on the caller stream, after the join
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    for mi, (d, k, mbs) in enumerate(mats):
        S[mi].check(f"S of matrix {mi}")
        want = np.zeros((d, r))
        for X, dY in mbs:
            want = O.sketch_accumulate(want, X.double().numpy(), dY.double().numpy(), 700 + mi, step, r)
        assert rel(copies[mi].cpu().numpy(), want) <= 1e-3, mi
