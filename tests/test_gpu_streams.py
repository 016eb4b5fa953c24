"""Calls on several CUDA streams at once: each (device, stream) has its own
workspace and counters, so interleaved sketches and applies of different
matrices on different streams must each match the oracle, exactly as when
issued alone."""
import numpy as np
import pytest

from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_S, TOL_V, TOL_DW = 1e-3, 1e-5, 1e-5


def rel(a, b):
    return np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b)


@pytest.fixture(scope="module")
def L():
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    return L


def test_three_streams_interleaved_match_oracle(L):
    import torch
    mats = [(264, 520, 96, 3), (1536, 776, 256, 3), (1032, 2056, 128, 3)]       # (d, k, r, seed)
    n, nmb = 640, 3
    streams = [torch.cuda.Stream() for _ in mats]
    state = []
    for i, (d, k, r, seed) in enumerate(mats):
        mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(40, i, mb))[:2]
               for mb in range(nmb)]
        dev = [(synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda()) for X, dY in mbs]
        S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
        W = torch.zeros((d, k), dtype=torch.float32, device="cuda")
        v = torch.zeros(d, dtype=torch.float32, device="cuda")
        norms = torch.zeros(2, dtype=torch.float64, device="cuda")
        state.append((d, k, r, seed + i, dev, S, W, v, norms))
    torch.cuda.synchronize()
    b2, eps, lr, c = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-5, 1.0))
    # microbatch-major order, so calls of the three matrices interleave on the device
    for mb in range(nmb):
        for st, (d, k, r, seed, dev, S, W, v, norms) in zip(streams, state):
            with torch.cuda.stream(st):
                L.logra_sketch_accumulate(dev[mb][0], dev[mb][1], S, seed, 9)
    for st, (d, k, r, seed, dev, S, W, v, norms) in zip(streams, state):
        with torch.cuda.stream(st):
            L.logra_rowadam_apply(W, S, v, seed, 9, b2, eps, lr, c, norms)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    for d, k, r, seed, dev, S, W, v, norms in state:
        S_or = np.zeros((d, r))
        for X, dY in dev:
            S_or = O.sketch_accumulate(S_or, X.double().cpu().numpy(), dY.double().cpu().numpy(), seed, 9, r)
        S_k = S.double().cpu().numpy()
        assert rel(S_k, S_or) <= TOL_S
        # apply checked on the kernel's own S, as in the stage-wise parity test
        _, v_or, n_or, dW_or = O.rowadam_apply(np.zeros((d, k)), S_k, np.zeros(d), seed, 9, b2, eps, lr, c)
        assert rel(v.double().cpu().numpy(), v_or) <= TOL_V
        assert rel(W.double().cpu().numpy(), dW_or) <= TOL_DW
        nr = norms.cpu().numpy()
        assert abs(nr[0] - n_or[0]) <= TOL_V * n_or[0] and abs(nr[1] - n_or[1]) <= TOL_V * n_or[1]


def test_microbatches_of_one_matrix_on_several_streams(L):
    """Microbatch calls that add into the same S, issued on four streams at once (bf16 and fp32
    paths): the atomic updates of S give the oracle's sum up to its tolerance."""
    import torch
    for dtype, (n, d, k, r), tol in (("bf16", (1024, 520, 1032, 128), 1e-3), ("f32", (257, 64, 72, 32), 1e-5)):
        mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(8, mb))[:2] for mb in range(8)]
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        dev = [(torch.from_numpy(X).to(tdt).cuda(), torch.from_numpy(dY).to(tdt).cuda()) for X, dY in mbs]
        S = torch.zeros((d, r), device="cuda")
        main = torch.cuda.current_stream()
        sts = [torch.cuda.Stream() for _ in range(4)]
        for st in sts:
            st.wait_stream(main)
        for i, (X, dY) in enumerate(dev):
            with torch.cuda.stream(sts[i % 4]):
                L.logra_sketch_accumulate(X, dY, S, 21, 3)
        for st in sts:
            main.wait_stream(st)
        torch.cuda.synchronize()
        assert L.logra_get_status() == 0
        S_or = np.zeros((d, r))
        for X, dY in dev:
            S_or = O.sketch_accumulate(S_or, X.double().cpu().numpy(), dY.double().cpu().numpy(), 21, 3, r)
        err = np.linalg.norm(S.double().cpu().numpy() - S_or) / np.linalg.norm(S_or)
        assert err <= tol, (dtype, err)


@pytest.mark.parametrize("streams", [2, 4, 16])
def test_concurrency_hint_changes_launches_not_results(L, streams):
    """The concurrency hint only reshapes the accumulate's grid: the sketch still equals the oracle."""
    import torch
    n, d, k, r = 2048, 1032, 520, 256
    mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(9, streams, mb))[:2]
           for mb in range(2)]
    L.logra_set_concurrency(streams)
    try:
        S = torch.zeros((d, r), device="cuda")
        S_or = np.zeros((d, r))
        for X, dY in mbs:
            Xb, dYb = synth.to_bf16_bits(X), synth.to_bf16_bits(dY)
            L.logra_sketch_accumulate(Xb.cuda(), dYb.cuda(), S, 31, 2)
            S_or = O.sketch_accumulate(S_or, Xb.double().numpy(), dYb.double().numpy(), 31, 2, r)
        torch.cuda.synchronize()
    finally:
        L.logra_set_concurrency(1)
    assert L.logra_get_status() == 0
    assert rel(S.double().cpu().numpy(), S_or) <= 1e-3
