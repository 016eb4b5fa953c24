"""CUDA-graph capture of sketch calls, and run-to-run spread of S.

Capture: the projection reduce-adds into a zeroed scratch buffer, and eager
calls skip the memset when the previous sketch on the stream left it zero.  A
graph is replayed later, after other work may have reused the workspace, so
captured calls must clear it themselves.  The test captures sketch calls,
runs an eager apply on the same stream (which overwrites the workspace),
replays, and compares with the oracle; then eager sketches on that stream
must still be right.

Spread: partial sums are added by TMA reduce-adds whose order depends on CTA
timing, so S is not bit-reproducible; two identical calls must agree far
inside the 1e-3 parity tolerance.
"""
import numpy as np
import pytest

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


def _mbs(n, d, k, count, key):
    out = []
    for mb in range(count):
        X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(key, mb))
        out.append((synth.to_bf16_bits(X), synth.to_bf16_bits(dY)))
    return out


def _oracle(mbs, d, r, seed, step):
    S = np.zeros((d, r))
    for X, dY in mbs:
        S = O.sketch_accumulate(S, X.double().numpy(), dY.double().numpy(), seed, step, r)
    return S


def test_captured_sketch_replays_after_eager_apply(L):
    import torch
    # n = 1024 (8 token tiles), k = 1032 (17 k-chunks): the projection's stream-K
    # ranges cut k ranges, so its partial segments reduce-add into the scratch
    n, d, k, r, seed, step = 1024, 264, 1032, 128, 71, 2
    L.logra_set_concurrency(1)
    mbs = _mbs(n, d, k, 2, 61)
    dev = [(X.cuda(), dY.cuda()) for X, dY in mbs]
    want = _oracle(mbs, d, r, seed, step)
    s = torch.cuda.Stream()
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    W = torch.zeros((512, 776), dtype=torch.float32, device="cuda")
    Sa = torch.randn((512, r), device="cuda") * 1e-3
    va = torch.zeros(512, device="cuda")
    with torch.cuda.stream(s):
        L.logra_reserve_workspace(max(L.lib().logra_sketch_workspace_bytes(n, d, k, r, 1),
                                      L.lib().logra_apply_workspace_bytes(512, 776, r)))
        for X, dY in dev:                                   # eager: leaves the scratch known-zero
            L.logra_sketch_accumulate(X, dY, S, seed, step)
        torch.cuda.synchronize()
        assert rel(S.cpu().numpy(), want) <= 1e-3
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            S.zero_()
            for X, dY in dev:
                L.logra_sketch_accumulate(X, dY, S, seed, step)
        for rep in range(3):
            L.logra_rowadam_apply(W, Sa, va, 5, rep, 0.999, 1e-8, 1e-5, 1.0)   # overwrites the workspace
            S.fill_(7.0)
            g.replay()
            torch.cuda.synchronize()
            assert rel(S.cpu().numpy(), want) <= 1e-3, rep
        # eager calls on the stream after the capture
        L.logra_rowadam_apply(W, Sa, va, 5, 9, 0.999, 1e-8, 1e-5, 1.0)
        S.zero_()
        for X, dY in dev:
            L.logra_sketch_accumulate(X, dY, S, seed, step)
        g.replay()
        S2 = torch.zeros_like(S)
        for X, dY in dev:
            L.logra_sketch_accumulate(X, dY, S2, seed, step)
        torch.cuda.synchronize()
    assert rel(S.cpu().numpy(), want) <= 1e-3
    assert rel(S2.cpu().numpy(), want) <= 1e-3
    assert L.logra_get_status() == 0


@pytest.mark.parametrize("n,d,k,r", [(8192, 5120, 5120, 256), (4096, 3584, 1024, 512)])
def test_sketch_run_to_run_spread(L, n, d, k, r):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(n + d + k + r)
    X = torch.randn((n, k), device="cuda", generator=g).to(torch.bfloat16)
    dY = (torch.randn((n, d), device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
    outs = []
    for _ in range(3):
        S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
        L.logra_sketch_accumulate(X, dY, S, 8, 8)
        outs.append(S)
    torch.cuda.synchronize()
    base = outs[0].double()
    for S in outs[1:]:
        spread = float((S.double() - base).norm() / base.norm())
        assert spread <= 1e-6, spread
    assert L.logra_get_status() == 0
