"""Seeded random shapes through the sketch and the apply, against the oracle.

Each case draws n (1..1100 tokens), d and k (multiples of 8 up to ~1100) and r (a multiple of 32 in
[32, 512]) so that token tiles, k chunks, d tiles, rank chunks and the stream-K segment boundaries
all fall at ragged places; the same seeds give the same cases on every run.  Every output (S, W,
its bf16 copy, v, the sync sketch, the norms) lies between guard regions that must come back
unchanged (tests/canary.py).
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
    return np.linalg.norm(np.asarray(a) - np.asarray(b)) / (nb if nb > 0 else 1.0)


def _case(i):
    g = np.random.default_rng(1000 + i)
    n = int(g.integers(1, 1100))
    d = 8 * int(g.integers(1, 140))
    k = 8 * int(g.integers(1, 140))
    r = 32 * int(g.integers(1, 17))
    return n, d, k, r


@pytest.mark.parametrize("i", range(24))
def test_random_shape_sketch_then_apply(L, i):
    import torch
    n, d, k, r = _case(i)
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(11, i))
    Xb, dYb = synth.to_bf16_bits(X), synth.to_bf16_bits(dY)
    gS = Guarded((d, r), torch.float32, fill=0.0)
    S = gS.t
    L.logra_sketch_accumulate(Xb.cuda(), dYb.cuda(), S, 500 + i, i)
    gS.check("S")
    S_or = O.sketch_accumulate(np.zeros((d, r)), Xb.double().numpy(), dYb.double().numpy(), 500 + i, i, r)
    Sg = S.double().cpu().numpy()
    assert rel(Sg, S_or) <= 1e-3, (n, d, k, r)
    # apply on the kernel's own S (stage-wise), W0 = 0 so that W = dW
    gW = Guarded((d, k), torch.float32, fill=0.0)
    gWb = Guarded((d, k), torch.bfloat16)
    gsync = Guarded((d, r), torch.float32)
    v0 = np.full(d, 1e-12, dtype=np.float32)
    gv = Guarded((d,), torch.float32, fill=torch.from_numpy(v0).cuda())
    gn = Guarded((2,), torch.float64, fill=0.0)
    W, v, norms = gW.t, gv.t, gn.t
    b2, eps, lr = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-5))
    L.logra_rowadam_apply_ex(W, S, v, 500 + i, i, b2, eps, lr, 1.0, norms, gWb.t, gsync.t)
    for g, what in ((gW, "W"), (gWb, "W bf16"), (gsync, "sync sketch"), (gv, "v"), (gn, "norms"), (gS, "S")):
        g.check(what)
    assert torch.equal(gWb.t, W.to(torch.bfloat16))
    assert L.logra_get_status() == 0
    _, v_or, n_or, dW_or = O.rowadam_apply(np.zeros((d, k)), Sg, v0.astype(np.float64), 500 + i, i, b2, eps, lr, 1.0)
    assert rel(v.double().cpu().numpy(), v_or) <= 1e-5, (n, d, k, r)
    assert rel(W.double().cpu().numpy(), dW_or) <= 1e-5, (n, d, k, r)
    nr = norms.cpu().numpy()
    assert abs(nr[1] - n_or[1]) <= 1e-5 * n_or[1], (n, d, k, r)
    assert rel(gsync.t.double().cpu().numpy(), O.sync_sketch(Sg, v_or, eps, lr, 1.0)) <= 1e-5, (n, d, k, r)
