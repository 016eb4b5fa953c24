"""Full-size parity on sampled outputs, in the launch configuration the bench times.

At the workloads' real shapes (27B-class and 7B-class projections, 8192-token
microbatches, r in {128, 256, 512}) the oracle cannot form the whole sketch or
the whole update quickly, but every column of S and every row of W is an
independent function of the inputs: the test checks seeded samples of them
one by one, plus properties that hold at any size.
"""
import numpy as np
import pytest

from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_S, TOL_ROW = 1e-3, 1e-5


@pytest.fixture(scope="module")
def L():
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    return L


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


CASES = [
    # (label, d, k, r, microbatches, mask)
    ("27b-gate", 27648, 5120, 256, 2, 0.30),
    ("27b-down", 5120, 27648, 256, 2, 0.30),
    ("27b-kv-r512", 1024, 5120, 512, 2, 0.30),
    ("27b-q-r128", 5120, 5120, 128, 2, 0.30),
    ("7b-up", 18944, 3584, 256, 2, 0.25),
]


@pytest.mark.parametrize("label,d,k,r,mbs,mask", CASES, ids=[c[0] for c in CASES])
def test_fullsize_sampled_sketch_and_apply(L, label, d, k, r, mbs, mask):
    import torch
    n = 8192
    seed, step = synth.matrix_seed(2026, 3, 5), 7
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    cols = np.random.default_rng(d + k + r).choice(r, size=3, replace=False)
    want_cols = np.zeros((d, len(cols)))
    for mb in range(mbs):
        X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=mask, key=(9, d, k, mb))
        Xb, dYb = synth.to_bf16_bits(X), synth.to_bf16_bits(dY)
        del X, dY
        L.logra_sketch_accumulate(Xb.cuda(), dYb.cuda(), S, seed, step)
        want_cols += O.sketch_columns(Xb.double().numpy(), dYb.double().numpy(), seed, step, r, cols)
        del Xb, dYb
    torch.cuda.synchronize()
    Sg = S.double().cpu().numpy()
    assert np.all(np.isfinite(Sg))
    assert rel(Sg[:, cols], want_cols) <= TOL_S

    # apply on the GPU's own S; sampled rows against the oracle's row-wise RowAdam
    W = torch.zeros((d, k), dtype=torch.float32, device="cuda")
    Wb = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
    v0 = np.full(d, 1e-12, dtype=np.float32)
    v = torch.from_numpy(v0).cuda()
    norms = torch.zeros(2, dtype=torch.float64, device="cuda")
    b2, eps, lr, c = (float(np.float32(x)) for x in (synth.BETA2, synth.EPS, synth.LR, 0.5))
    L.logra_rowadam_apply_ex(W, S, v, seed, step, b2, eps, lr, c, norms, Wb, None)
    torch.cuda.synchronize()
    rows = np.random.default_rng(d * 3 + k).choice(d, size=6, replace=False)
    v_or, dW_or, _ = O.rowadam_rows(Sg[rows], v0[rows].astype(np.float64), k, seed, step, b2, eps, lr, c)
    assert rel(v.double().cpu().numpy()[rows], v_or) <= TOL_ROW
    Wr = W[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    assert rel(Wr, dW_or) <= TOL_ROW
    # properties at any size: ||S||^2 is the norm of the kernel's S; the bf16 copy is RN(W)
    nr = norms.cpu().numpy()
    # the kernel sums squares of S in fp32 over 32-column blocks, then in fp64:
    # worst-case relative error 32 * 2^-24 (~1.9e-6), inside the 1e-5 norm tolerance
    assert abs(nr[0] - float(np.sum(Sg * Sg))) <= 2e-6 * nr[0]
    assert torch.equal(Wb, W.to(torch.bfloat16))
    # ||dW||^2 identity: (lr c)^2 sum_i k m_i / (v_i + eps), with m_i from the kernel's v
    vg = v.double().cpu().numpy()
    m = (vg - b2 * v0.astype(np.float64)) / (1.0 - b2)
    want_dw2 = (lr * c) ** 2 * float(np.sum(k * m / (vg + eps)))
    assert abs(nr[1] - want_dw2) <= 1e-4 * want_dw2


HINT_CASES = [
    # (label, d, k, r): shapes the bench's multi-matrix steps issue on 16 streams
    ("7b-gate", 18944, 3584, 256),
    ("7b-down", 3584, 18944, 256),
    ("7b-k", 512, 3584, 256),
    ("27b-gate", 27648, 5120, 256),
    ("27b-kv-r512", 1024, 5120, 512),
]


@pytest.mark.parametrize("label,d,k,r", HINT_CASES, ids=[c[0] for c in HINT_CASES])
def test_fullsize_sampled_sketch_in_the_benchs_launch_shape(L, label, d, k, r):
    """The step's launch shape: concurrency hint 16, so the projection runs one CTA per 256-token
    group over the whole k range and writes the accumulate's image itself, and the accumulate
    takes fewer, longer CTA-pair ranges.  Sampled columns of S against the oracle, 8192-token
    microbatches."""
    import torch
    n = 8192
    seed, step = synth.matrix_seed(2026, 11, 2), 4
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    cols = np.random.default_rng(d + 7 * k).choice(r, size=3, replace=False)
    want_cols = np.zeros((d, len(cols)))
    L.logra_set_concurrency(16)
    try:
        for mb in range(2):
            X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(10, d, k, mb))
            Xb, dYb = synth.to_bf16_bits(X), synth.to_bf16_bits(dY)
            del X, dY
            L.logra_sketch_accumulate(Xb.cuda(), dYb.cuda(), S, seed, step)
            want_cols += O.sketch_columns(Xb.double().numpy(), dYb.double().numpy(), seed, step, r, cols)
            del Xb, dYb
        torch.cuda.synchronize()
    finally:
        L.logra_set_concurrency(1)
    assert L.logra_get_status() == 0
    Sg = S.double().cpu().numpy()
    assert np.all(np.isfinite(Sg))
    assert rel(Sg[:, cols], want_cols) <= TOL_S
