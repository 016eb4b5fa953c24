"""Bit-exact checks of the sign generators the kernels themselves use.

`logra_sign_matrix` writes A explicitly, but the contractions never read that
matrix: the projection builds its sign tiles in shared memory, the apply and
the reconstruct build theirs in another layout, and the row-norm pass counts
sign words for the Gram matrix M = Sigma Sigma^T.  One-hot inputs make each of
those paths return entries of A (or of M) exactly, so they are compared bit
for bit with the oracle's fp32 A = Sigma * fl32(1/sqrt(r)) and integer M
(academy.dair.ai summary, "Gradient sketches": the random-sign projection is
redrawn per step and shared by the step's microbatches).

  * sketch:      token t with X_t = e_j and dY_t = e_t gives S[t, :] = A[:, j]
                 (P = X Sigma^T is exactly +-1, its low bf16 term 0, and the
                 scale fl32(1/sqrt(r)) multiplies +-1 exactly)
  * reconstruct: S rows e_b give (S A)[row, :] = A[b, :]
  * Gram:        S rows e_a + e_b with beta2 = 0 give v = (2k + 2 M_ab) / (r k),
                 from which the integer M_ab is recovered exactly

Also here: the bf16 accumulate form of the reconstruct (rollout weights are
bf16), exact for one-hot S and within one bf16 rounding for a realistic S.
Every output sits between guard regions (tests/canary.py).
"""
import numpy as np
import pytest

from canary import Guarded
from oracle import logra_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import torch
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    torch.cuda.init()
    return L


def _one_hot_rows(n, width, cols, dtype):
    import torch
    X = torch.zeros((n, width), dtype=dtype)
    X[torch.arange(n), torch.as_tensor(cols, dtype=torch.long)] = 1
    return X


# (r, k, tokens per call): k % 64 != 0 (a partial last sign word) and k over several 64-column
# chunks; r over the single-CTA accumulate (32, 96, 128, 384) and the CTA-pair one (256, 512).
SKETCH_CASES = [(32, 200, 1500), (96, 1000, 1500), (256, 4104, 1500), (384, 776, 600), (512, 2056, 600),
                (256, 27656, 1500), (256, 1032, 1500), (128, 520, 1500), (512, 776, 1500)]


@pytest.mark.parametrize("r,k,per", SKETCH_CASES)
def test_sketch_generator_bit_exact(L, r, k, per):
    import torch
    seed, step = 0x5EED0000 + r, 3 + k
    A = O.projection_matrix_fp32(seed, step, r, k)            # r x k fp32
    g = np.random.default_rng(r * 7 + k)
    # every column once (the last partial word included), in random order, up to 1500 per call
    cols = g.permutation(k)
    if k > 5000:
        cols = np.concatenate([cols[:1400], np.arange(k - 70, k)])
    for c0 in range(0, len(cols), per):
        J = cols[c0:c0 + per]
        n = len(J)
        d = ((n + 7) // 8) * 8 + 8
        X = _one_hot_rows(n, k, J, torch.bfloat16).cuda()
        dY = _one_hot_rows(n, d, np.arange(n), torch.bfloat16).cuda()
        S = Guarded((d, r), torch.float32, fill=0.0)
        L.logra_sketch_accumulate(X, dY, S.t, seed, step)
        S.check("S")
        got = S.t.cpu().numpy()
        want = np.ascontiguousarray(A[:, J].T)                # row t = column J[t] of A
        assert np.array_equal(got[:n].view(np.uint32), want.view(np.uint32)), (r, k, c0)
        assert not np.any(got[n:]), (r, k, c0)
    assert L.logra_get_status() == 0


@pytest.mark.parametrize("r,k", [(96, 1000), (256, 1032), (512, 520)])
def test_sketch_direct_image_bit_exact(L, r, k):
    """With calls on several streams (concurrency hint) and at least one 256-token group per stream
    share of the SMs, every projection CTA covers a whole k range and writes the accumulate's hi/lo
    image itself (no fp32 P^T, no split launch).  6000 tokens: token t takes column t mod k."""
    import torch
    seed, step = 0xD1EC7 + r, 2
    A = O.projection_matrix_fp32(seed, step, r, k)
    n = 6000
    J = np.arange(n) % k
    d = n + 8
    X = _one_hot_rows(n, k, J, torch.bfloat16).cuda()
    dY = _one_hot_rows(n, d, np.arange(n), torch.bfloat16).cuda()
    L.logra_set_concurrency(8)
    try:
        S = Guarded((d, r), torch.float32, fill=0.0)
        L.logra_sketch_accumulate(X, dY, S.t, seed, step)
        S.check("S")
    finally:
        L.logra_set_concurrency(1)
    got = S.t.cpu().numpy()
    want = np.ascontiguousarray(A[:, J].T)
    assert np.array_equal(got[:n].view(np.uint32), want.view(np.uint32))
    assert not np.any(got[n:])
    assert L.logra_get_status() == 0


@pytest.mark.parametrize("n,d,k,r", [(8192, 1032, 1544, 256), (5000, 264, 3080, 160), (6144, 2056, 520, 512)])
def test_sketch_direct_image_matches_oracle(L, n, d, k, r):
    """The direct-image projection on realistic inputs, two microbatches, against the oracle (1e-3)."""
    import torch
    from rank_gradient_sketching_02_gb300 import synth
    L.logra_set_concurrency(8)
    try:
        S = Guarded((d, r), torch.float32, fill=0.0)
        S_or = np.zeros((d, r))
        for mb in range(2):
            X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(71, n, mb))
            Xb, dYb = synth.to_bf16_bits(X), synth.to_bf16_bits(dY)
            L.logra_sketch_accumulate(Xb.cuda(), dYb.cuda(), S.t, 9, 4)
            S_or = O.sketch_accumulate(S_or, Xb.double().numpy(), dYb.double().numpy(), 9, 4, r)
        S.check("S")
    finally:
        L.logra_set_concurrency(1)
    got = S.t.double().cpu().numpy()
    assert np.linalg.norm(got - S_or) / np.linalg.norm(S_or) <= 1e-3
    assert L.logra_get_status() == 0


@pytest.mark.parametrize("r,k", [(32, 200), (96, 1000), (256, 4104), (384, 776), (512, 2056), (128, 18952)])
def test_reconstruct_generator_bit_exact(L, r, k):
    import torch
    seed, step = 0xA11CE + r, 11
    A = O.projection_matrix_fp32(seed, step, r, k)
    d = 2 * r + 8                                             # every rank twice, ragged row tile
    rows = np.arange(d) % r
    S = torch.zeros((d, r), dtype=torch.float32)
    S[torch.arange(d), torch.as_tensor(rows)] = 1.0
    S = S.cuda()
    out = Guarded((d, k), torch.float32)
    L.logra_reconstruct(S, k, seed, step, out.t)
    out.check("reconstruct fp32")
    got = out.t.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), A[rows].view(np.uint32))
    # accumulate into fp32: one fp32 rounding of base + A
    base = np.random.default_rng(r + k).standard_normal((d, k)).astype(np.float32)
    acc = Guarded((d, k), torch.float32, fill=torch.from_numpy(base).cuda())
    L.logra_reconstruct(S, k, seed, step, acc.t, accumulate=True)
    acc.check("reconstruct fp32 accumulate")
    assert np.array_equal(acc.t.cpu().numpy().view(np.uint32), (base + A[rows]).view(np.uint32))
    # accumulate into bf16: computed in fp32, rounded once to bf16
    base_b = torch.from_numpy(base).to(torch.bfloat16)
    accb = Guarded((d, k), torch.bfloat16, fill=base_b.cuda())
    L.logra_reconstruct(S, k, seed, step, accb.t, accumulate=True)
    accb.check("reconstruct bf16 accumulate")
    want_b = (base_b.float() + torch.from_numpy(A[rows])).to(torch.bfloat16)
    assert torch.equal(accb.t.cpu().view(torch.int16), want_b.view(torch.int16))
    assert L.logra_get_status() == 0


@pytest.mark.parametrize("r,k", [(32, 200), (96, 1000), (256, 4104), (384, 776), (512, 2056), (512, 27656)])
def test_gram_generator_exact_through_v(L, r, k):
    import torch
    seed, step = 0x6A4A + r, 5
    M = O.gram_matrix(seed, step, r, k)
    g = np.random.default_rng(r + 3 * k)
    # pairs a != b in every 32 x 32 tile of M (diagonal tiles included), plus random ones
    pairs = []
    for ta in range(r // 32):
        for tb in range(ta, r // 32):
            a = 32 * ta + int(g.integers(32))
            b = 32 * tb + int(g.integers(32))
            if a == b:
                b = 32 * tb + (b - 32 * tb + 1) % 32
            pairs.append((a, b))
    while len(pairs) % 8:
        a, b = g.choice(r, 2, replace=False)
        pairs.append((int(a), int(b)))
    d = len(pairs)
    S = torch.zeros((d, r), dtype=torch.float32)
    for i, (a, b) in enumerate(pairs):
        S[i, a] = 1.0
        S[i, b] = 1.0
    S = S.cuda()
    W = Guarded((d, k), torch.float32, fill=0.0)
    v = Guarded((d,), torch.float32, fill=0.0)
    L.logra_rowadam_apply(W.t, S, v.t, seed, step, 0.0, 1e-8, 1e-6, 1.0)
    W.check("W")
    v.check("v")
    vv = v.t.double().cpu().numpy()
    q = np.rint(vv * r * k)                                   # q = S_i M S_i^T = 2k + 2 M_ab, an integer
    assert np.all(np.abs(vv * r * k - q) < 1e-2)
    got = (q - 2 * k) / 2
    want = np.array([M[a, b] for a, b in pairs], dtype=np.float64)
    assert np.array_equal(got, want)
    assert L.logra_get_status() == 0


def test_reconstruct_bf16_accumulate_matches_oracle(L):
    """The rollout-weight path: bf16 weights += S' A from a realistic sync sketch."""
    import torch
    d, k, r = 264, 1544, 256
    g = np.random.default_rng(91)
    S32 = (g.standard_normal((d, r)) * 1e-3 * np.exp(g.standard_normal((d, 1)))).astype(np.float32)
    want_d = O.reconstruct(S32.astype(np.float64), 17, 4, k)
    scale = np.sqrt(np.mean(want_d ** 2))
    base = torch.from_numpy((g.standard_normal((d, k)) * 4 * scale).astype(np.float32)).to(torch.bfloat16)
    out = Guarded((d, k), torch.bfloat16, fill=base.cuda())
    L.logra_reconstruct(torch.from_numpy(S32).cuda(), k, 17, 4, out.t, accumulate=True)
    out.check("bf16 accumulate")
    got = out.t.cpu()
    want = (base.double() + torch.from_numpy(want_d)).to(torch.bfloat16)     # one rounding of the exact sum
    gv, wv = got.double().numpy(), want.double().numpy()
    # one bf16 rounding of a sum whose fp32 update term carries its own error (the sketch enters the
    # contraction as a two-term bf16 expansion, ~2^-16 relative per element, summed over r terms): within
    # one bf16 ulp of the correctly rounded exact sum, plus that term's error where the sum cancels
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(wv), 1e-30))) - 7)
    assert np.all(np.abs(gv - wv) <= ulp + 2e-4 * scale)
    assert np.mean(gv == wv) >= 0.99
    assert np.linalg.norm(gv - wv) / np.linalg.norm(wv) <= 1e-3
