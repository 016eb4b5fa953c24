"""Pins for the fp64 oracle, each against something other than the oracle itself.

* published SplitMix64 outputs (the sign generator's definition),
* pure-Python brute-force sums for the sketch and for RowAdam,
* G A^T with G formed explicitly (the sketch's defining identity),
* linearity over microbatches and invariance to padding rows,
* Monte-Carlo unbiasedness of S A with the closed-form error of the mean,
* RowAdam closed forms (first step from v = 0, two steps by hand, S = 0, c = 0,
  scale invariance at eps = 0) and the ||dW||^2 identity,
* the Gram identity ||(S A)_i||^2 = S_i (Sigma Sigma^T) S_i^T / r with the popcount form.

The last group plants mistakes in copies of oracle functions and checks that a
pin catches each one.
"""
import math
import os

import numpy as np
import pytest

from oracle import logra_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_words(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(int(line, 16))
    return out


# ---------------------------------------------------------------- generator
def test_splitmix64_published_outputs():
    want = _golden_words("splitmix64_seed0.txt")
    got = [int(x) for x in O.splitmix64_outputs(0, len(want))]
    assert got == want


def test_step_key_is_splitmix_output():
    want = _golden_words("splitmix64_seed0.txt")
    for step, w in enumerate(want):
        assert int(O.step_key(0, step)) == w


def _py_mix(z):
    z &= O.MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & O.MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & O.MASK64
    return z ^ (z >> 31)


def test_sign_matrix_bit_layout_python_ints():
    # Same reading in unbounded Python integers: catches numpy casting/shift slips.
    seed, step, r, k = 0x1234_5678_9ABC, 7, 5, 200
    key = _py_mix(seed + (step + 1) * 0x9E3779B97F4A7C15)
    Sg = O.sign_matrix(seed, step, r, k)
    for i in range(r):
        for j in range(k):
            word = _py_mix(key ^ ((i << 32) | (j // 64)))
            want = -1 if (word >> (j % 64)) & 1 else 1
            assert Sg[i, j] == want


def test_sign_matrix_statistics_and_redraw():
    r, k = 64, 4096
    Sg = O.sign_matrix(3, 11, r, k).astype(np.float64)
    assert set(np.unique(Sg)) == {-1.0, 1.0}
    assert abs(Sg.mean()) < 4.0 / math.sqrt(r * k)
    # rows look independent: off-diagonal Gram entries ~ N(0, k)
    M = Sg @ Sg.T
    off = M[~np.eye(r, dtype=bool)]
    assert np.all(np.diag(M) == k)
    assert abs(off.mean()) < 4.0 * math.sqrt(k) / math.sqrt(off.size / 2)
    assert 0.8 < off.var() / k < 1.2
    # held fixed within a step, redrawn across steps (and across seeds)
    assert np.array_equal(O.sign_matrix(3, 11, r, k), O.sign_matrix(3, 11, r, k))
    assert np.mean(O.sign_matrix(3, 12, r, k) == O.sign_matrix(3, 11, r, k)) < 0.52
    assert np.mean(O.sign_matrix(4, 11, r, k) == O.sign_matrix(3, 11, r, k)) < 0.52


@pytest.mark.parametrize("r", [32, 128, 256, 512])
def test_projection_fp32_values(r):
    A32 = O.projection_matrix_fp32(1, 2, r, 130)
    s = np.float32(1.0 / math.sqrt(r))
    assert A32.dtype == np.float32
    assert set(np.unique(np.abs(A32))) == {s}
    A = O.projection_matrix(1, 2, r, 130)
    np.testing.assert_allclose(A * A, 1.0 / r, rtol=1e-15)


# ---------------------------------------------------------------- sketch
def _tiny(n=5, d=3, k=70, seed=1):
    g = np.random.default_rng(seed)
    return g.standard_normal((n, k)), g.standard_normal((n, d))


def test_sketch_brute_force_loops():
    n, d, k, r = 5, 3, 70, 4
    X, dY = _tiny(n, d, k)
    seed, step = 9, 2
    Sg = O.sign_matrix(seed, step, r, k)
    S = O.sketch_accumulate(np.zeros((d, r)), X, dY, seed, step, r)
    for a in range(d):
        for b in range(r):
            acc = 0.0
            for t in range(n):
                for j in range(k):
                    acc += dY[t, a] * X[t, j] * float(Sg[b, j])
            acc /= math.sqrt(r)
            assert abs(S[a, b] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_sketch_equals_full_gradient_times_At():
    n, d, k, r = 33, 17, 150, 8
    X, dY = _tiny(n, d, k, seed=2)
    G = dY.T @ X                                   # d x k, formed only in the test
    A = O.projection_matrix(5, 0, r, k)
    want = G @ A.T
    got = O.sketch_accumulate(np.zeros((d, r)), X, dY, 5, 0, r)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert got.shape == (d, r)


def test_sketch_linear_over_microbatches():
    d, k, r = 12, 96, 16
    g = np.random.default_rng(3)
    mbs = [(g.standard_normal((n, k)), g.standard_normal((n, d))) for n in (7, 1, 20, 13)]
    S = np.zeros((d, r))
    for X, dY in mbs:
        S = O.sketch_accumulate(S, X, dY, 4, 1, r)
    Xc = np.concatenate([m[0] for m in mbs])
    dYc = np.concatenate([m[1] for m in mbs])
    S1 = O.sketch_accumulate(np.zeros((d, r)), Xc, dYc, 4, 1, r)
    np.testing.assert_allclose(S, S1, rtol=1e-12, atol=1e-12)


def test_sketch_of_stacked_two_term_planes():
    """The identity the fp32-input path rests on: with x = x1 + x2 + e (x1 = RN_bf16(x),
    x2 = RN_bf16(x - x1), |e| <= u^2 |x| for bf16's unit roundoff u = 2^-8), the sketch of the
    token-stacked planes [X1; X2; X1; X2] against [dY1; dY1; dY2; dY2] is the sketch of
    (X1 + X2, dY1 + dY2), and that is well inside the fp32 bound (1e-5) of the sketch of the
    fp32 inputs themselves."""
    import torch
    n, d, k, r = 48, 24, 136, 32
    g = np.random.default_rng(12)
    X = g.standard_normal((n, k)).astype(np.float32)
    dY = (g.standard_normal((n, d)) * np.exp(-7 + 1.5 * g.standard_normal((n, 1)))).astype(np.float32)

    def planes(a):
        t = torch.from_numpy(a)
        hi = t.to(torch.bfloat16).float()
        lo = (t - hi).to(torch.bfloat16).float()      # t - hi is exact in fp32
        return hi.double().numpy(), lo.double().numpy()

    X1, X2 = planes(X)
    dY1, dY2 = planes(dY)
    stacked = O.sketch_accumulate(np.zeros((d, r)), np.concatenate([X1, X2, X1, X2]),
                                  np.concatenate([dY1, dY1, dY2, dY2]), 9, 2, r)
    summed = O.sketch_accumulate(np.zeros((d, r)), X1 + X2, dY1 + dY2, 9, 2, r)
    exact = O.sketch_accumulate(np.zeros((d, r)), X.astype(np.float64), dY.astype(np.float64), 9, 2, r)
    np.testing.assert_allclose(stacked, summed, rtol=1e-12, atol=1e-12 * np.abs(summed).max())
    assert np.all(np.abs(X1 + X2 - X) <= 2.0 ** -16 * np.abs(X))
    assert np.all(np.abs(dY1 + dY2 - dY) <= 2.0 ** -16 * np.abs(dY))
    err = np.linalg.norm(summed - exact) / np.linalg.norm(exact)
    assert 0 < err <= 1e-5, err
    # one plane alone (bf16 inputs) is two orders worse: the second plane carries the fp32 accuracy
    one = O.sketch_accumulate(np.zeros((d, r)), X1, dY1, 9, 2, r)
    assert np.linalg.norm(one - exact) / np.linalg.norm(exact) > 100 * err


def test_sketch_padding_rows_contribute_nothing():
    n, d, k, r = 40, 9, 128, 8
    X, dY = _tiny(n, d, k, seed=4)
    keep = np.ones(n, bool)
    keep[[0, 5, 6, 39]] = False
    Xm, dYm = X.copy(), dY.copy()
    Xm[~keep] = 0
    dYm[~keep] = 0
    a = O.sketch_accumulate(np.zeros((d, r)), Xm, dYm, 1, 1, r)
    b = O.sketch_accumulate(np.zeros((d, r)), X[keep], dY[keep], 1, 1, r)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_input_gradient_brute_force_loops():
    n, d, k = 4, 6, 5
    X, dY = _tiny(n, d, k, seed=11)
    W = np.random.default_rng(12).standard_normal((d, k))
    got = O.input_gradient(dY, W)
    for t in range(n):
        for j in range(k):
            acc = 0.0
            for a in range(d):
                acc += dY[t, a] * W[a, j]
            assert abs(got[t, j] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_linear_backward_matches_autograd_of_the_layer():
    """dX is what autograd gives for Y = X W^T, and the sketch is the autograd
    weight gradient times A^T (S = G A^T with G from the layer itself)."""
    torch = pytest.importorskip("torch")
    n, d, k, r = 19, 13, 136, 32
    X, dY = _tiny(n, d, k, seed=13)
    W = np.random.default_rng(14).standard_normal((d, k))
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.linear(Xt, Wt).backward(torch.tensor(dY, dtype=torch.float64))
    S0 = np.random.default_rng(15).standard_normal((d, r))
    dX, S = O.linear_backward(S0, X, dY, W, 6, 2, r)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-12, atol=1e-12)
    A = O.projection_matrix(6, 2, r, k)
    np.testing.assert_allclose(S - S0, Wt.grad.numpy() @ A.T, rtol=1e-10, atol=1e-10)


def test_sketch_columns_match_full():
    n, d, k, r = 21, 11, 200, 32
    X, dY = _tiny(n, d, k, seed=5)
    S = O.sketch_accumulate(np.zeros((d, r)), X, dY, 8, 3, r)
    cols = [0, 7, 31]
    np.testing.assert_allclose(O.sketch_columns(X, dY, 8, 3, r, cols), S[:, cols],
                               rtol=1e-12, atol=1e-12)


def test_reconstruction_unbiased_monte_carlo():
    # E[A^T A] = I, so the mean of S A over independent draws converges to G with
    # E||mean - G||_F^2 = (k-1) ||G||_F^2 / (r T)  (off-diagonal (A^T A)_jj' have
    # variance 1/r and are pairwise uncorrelated).
    d, k, r, T = 8, 64, 8, 3000
    g = np.random.default_rng(6)
    G = g.standard_normal((d, k))
    acc = np.zeros((d, k))
    for step in range(T):
        A = O.projection_matrix(77, step, r, k)
        S = G @ A.T
        acc += O.reconstruct(S, 77, step, k)
    mean = acc / T
    err2 = np.sum((mean - G) ** 2)
    expect = (k - 1) * np.sum(G * G) / (r * T)
    assert 0.8 < err2 / expect < 1.2, err2 / expect


# ---------------------------------------------------------------- RowAdam
def _brute_ghat(S, Sg, r):
    d, k = S.shape[0], Sg.shape[1]
    out = [[0.0] * k for _ in range(d)]
    for i in range(d):
        for j in range(k):
            out[i][j] = sum(S[i, b] * float(Sg[b, j]) for b in range(r)) / math.sqrt(r)
    return out


def test_rowadam_first_step_closed_form():
    d, k, r = 4, 66, 8
    g = np.random.default_rng(7)
    S = g.standard_normal((d, r)) * 1e-2
    W = g.standard_normal((d, k)) * 0.02
    beta2, eps, lr, c = 0.999, 1e-8, 1e-5, 0.7
    Wn, vn, norms, dW = O.rowadam_apply(W, S, np.zeros(d), 2, 5, beta2, eps, lr, c)
    Gh = _brute_ghat(S, O.sign_matrix(2, 5, r, k), r)
    for i in range(d):
        m = sum(x * x for x in Gh[i]) / k
        assert abs(vn[i] - (1 - beta2) * m) <= 1e-13 * m
        den = math.sqrt((1 - beta2) * m + eps)
        for j in range(k):
            want = -lr * c * Gh[i][j] / den
            assert abs(dW[i, j] - want) <= 1e-12 * abs(lr * c * Gh[i][j] / den) + 1e-300
            assert abs(Wn[i, j] - (W[i, j] + want)) <= 1e-15
    assert abs(norms[0] - float(np.sum(S * S))) <= 1e-15 * norms[0]


def test_rowadam_two_steps_by_hand():
    d, k, r = 3, 64, 4
    g = np.random.default_rng(8)
    S0, S1 = g.standard_normal((d, r)), g.standard_normal((d, r))
    beta2, eps, lr, c = 0.9, 1e-6, 1e-3, 1.0
    W0 = np.zeros((d, k))
    W1, v1, _, _ = O.rowadam_apply(W0, S0, np.zeros(d), 1, 0, beta2, eps, lr, c)
    W2, v2, _, dW2 = O.rowadam_apply(W1, S1, v1, 1, 1, beta2, eps, lr, c)
    G0 = np.array(_brute_ghat(S0, O.sign_matrix(1, 0, r, k), r))
    G1 = np.array(_brute_ghat(S1, O.sign_matrix(1, 1, r, k), r))
    m0 = (G0 ** 2).mean(1)
    m1 = (G1 ** 2).mean(1)
    v1h = (1 - beta2) * m0
    v2h = beta2 * v1h + (1 - beta2) * m1
    np.testing.assert_allclose(v2, v2h, rtol=1e-13)
    W2h = -lr * c * (G0 / np.sqrt(v1h + eps)[:, None] + G1 / np.sqrt(v2h + eps)[:, None])
    np.testing.assert_allclose(W2, W2h, rtol=1e-12, atol=1e-18)


def test_rowadam_zero_sketch_and_zero_scale():
    d, k, r = 5, 128, 8
    g = np.random.default_rng(9)
    W = g.standard_normal((d, k))
    v = np.abs(g.standard_normal(d))
    Wn, vn, norms, dW = O.rowadam_apply(W, np.zeros((d, r)), v, 0, 0, 0.99, 1e-8, 1e-3, 1.0)
    assert np.all(dW == 0) and np.array_equal(Wn, W)
    np.testing.assert_allclose(vn, 0.99 * v, rtol=1e-15)
    assert norms[0] == 0 and norms[1] == 0
    S = g.standard_normal((d, r))
    Wn, vn, norms, dW = O.rowadam_apply(W, S, v, 0, 0, 0.99, 1e-8, 1e-3, 0.0)
    assert np.array_equal(Wn, W) and norms[1] == 0
    Wn1, vn1, _, _ = O.rowadam_apply(W, S, v, 0, 0, 0.99, 1e-8, 1e-3, 1.0)
    np.testing.assert_allclose(vn, vn1, rtol=1e-15)   # v still advances when c = 0


def test_rowadam_scale_invariant_at_eps0():
    d, k, r = 6, 128, 16
    S = np.random.default_rng(10).standard_normal((d, r))
    _, _, _, dW1 = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 3, 3, 0.999, 0.0, 1e-2, 1.0)
    _, _, _, dW2 = O.rowadam_apply(np.zeros((d, k)), 1e4 * S, np.zeros(d), 3, 3, 0.999, 0.0, 1e-2, 1.0)
    np.testing.assert_allclose(dW1, dW2, rtol=1e-12)


def test_update_norm_identity():
    d, k, r = 7, 192, 16
    g = np.random.default_rng(11)
    S, v = g.standard_normal((d, r)), np.abs(g.standard_normal(d))
    lr, c, eps = 1e-3, 0.5, 1e-8
    _, vn, norms, _ = O.rowadam_apply(np.zeros((d, k)), S, v, 1, 2, 0.95, eps, lr, c)
    m = np.mean(O.reconstruct(S, 1, 2, k) ** 2, axis=1)
    np.testing.assert_allclose(norms[1], (lr * c) ** 2 * np.sum(k * m / (vn + eps)), rtol=1e-12)


def test_sync_sketch_rebuilds_applied_update():
    d, k, r = 9, 256, 32
    g = np.random.default_rng(12)
    S, v = g.standard_normal((d, r)), np.abs(g.standard_normal(d)) * 1e-3
    _, vn, _, dW = O.rowadam_apply(np.zeros((d, k)), S, v, 4, 4, 0.999, 1e-8, 1e-5, 0.9)
    Sp = O.sync_sketch(S, vn, 1e-8, 1e-5, 0.9)
    np.testing.assert_allclose(O.reconstruct(Sp, 4, 4, k), dW, rtol=1e-12, atol=1e-20)


def test_rowadam_rows_match_full():
    d, k, r = 10, 128, 8
    g = np.random.default_rng(13)
    S, v = g.standard_normal((d, r)), np.abs(g.standard_normal(d))
    _, vn, _, dW = O.rowadam_apply(np.zeros((d, k)), S, v, 6, 1, 0.99, 1e-8, 1e-3, 1.0)
    rows = [0, 4, 9]
    vr, dWr, _ = O.rowadam_rows(S[rows], v[rows], k, 6, 1, 0.99, 1e-8, 1e-3, 1.0)
    np.testing.assert_allclose(vr, vn[rows], rtol=1e-14)
    np.testing.assert_allclose(dWr, dW[rows], rtol=1e-14)


# ---------------------------------------------------------------- bias-corrected variant
def test_bias_corrected_first_step_has_unit_rms_rows():
    """From v = 0 with eps = 0, the first corrected step (t = 1) divides each row of Ghat by
    its own rms, whatever beta2: ||dW_i||^2 = (lr c)^2 k exactly (uncorrected it is that
    over 1 - beta2), and the stored v keeps its uncorrected value."""
    d, k, r = 5, 192, 16
    S = np.random.default_rng(40).standard_normal((d, r)) * np.array([[1e-4], [1e-2], [1.0], [3.0], [1e3]])
    lr, c = 1e-3, 0.6
    for beta2 in (0.9, 0.999, 0.99999):
        _, vn, norms, dW = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 2, 3, beta2, 0.0, lr, c, t=1)
        np.testing.assert_allclose(np.sum(dW * dW, axis=1), (lr * c) ** 2 * k, rtol=1e-12)
        np.testing.assert_allclose(norms[1], d * (lr * c) ** 2 * k, rtol=1e-12)
        m = np.mean(np.array(_brute_ghat(S, O.sign_matrix(2, 3, r, k), r)) ** 2, axis=1)
        np.testing.assert_allclose(vn, (1 - beta2) * m, rtol=1e-12)
        _, _, _, dW0 = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 2, 3, beta2, 0.0, lr, c)
        np.testing.assert_allclose(np.sum(dW0 * dW0, axis=1), (lr * c) ** 2 * k / (1 - beta2), rtol=1e-10)


def test_bias_corrected_constant_gradient_same_step_every_t():
    """A constant gradient from v = 0: v_t = (1 - beta2^t) m, so the corrected v is m at
    every t and every step is the same; without correction the steps shrink."""
    d, k, r = 4, 128, 8
    S = np.random.default_rng(41).standard_normal((d, r))
    beta2, eps, lr = 0.9, 0.0, 1e-2
    v = np.zeros(d)
    steps = []
    for t in range(1, 6):
        _, v, _, dW = O.rowadam_apply(np.zeros((d, k)), S, v, 7, 0, beta2, eps, lr, 1.0, t=t)
        steps.append(dW)
    for dW in steps[1:]:
        np.testing.assert_allclose(dW, steps[0], rtol=1e-12)
    _, _, _, late = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 7, 0, beta2, eps, lr, 1.0, t=10**6)
    _, _, _, plain = O.rowadam_apply(np.zeros((d, k)), S, np.zeros(d), 7, 0, beta2, eps, lr, 1.0)
    np.testing.assert_allclose(late, plain, rtol=1e-12)   # 1 - beta2^t -> 1


def test_bias_corrected_sync_sketch_and_rows():
    d, k, r = 6, 256, 16
    g = np.random.default_rng(42)
    S, v = g.standard_normal((d, r)), np.abs(g.standard_normal(d)) * 1e-2
    _, vn, _, dW = O.rowadam_apply(np.zeros((d, k)), S, v, 4, 4, 0.99, 1e-8, 1e-4, 0.9, t=3)
    Sp = O.sync_sketch(S, vn, 1e-8, 1e-4, 0.9, beta2=0.99, t=3)
    np.testing.assert_allclose(O.reconstruct(Sp, 4, 4, k), dW, rtol=1e-12, atol=1e-20)
    vr, dWr, _ = O.rowadam_rows(S[[1, 4]], v[[1, 4]], k, 4, 4, 0.99, 1e-8, 1e-4, 0.9, t=3)
    np.testing.assert_allclose(dWr, dW[[1, 4]], rtol=1e-14)


# ---------------------------------------------------------------- Gram identity
@pytest.mark.parametrize("k", [64, 200, 640])
def test_gram_identity_and_popcount(k):
    r = 16
    M = O.gram_matrix(5, 9, r, k)
    words = O.sign_words(5, 9, r, k)
    nw = words.shape[1]
    valid = [((1 << 64) - 1) if (w + 1) * 64 <= k else ((1 << (k - 64 * w)) - 1) for w in range(nw)]
    for a in range(r):
        for b in range(r):
            diff = sum(bin((int(words[a, w]) ^ int(words[b, w])) & valid[w]).count("1")
                       for w in range(nw))
            assert M[a, b] == k - 2 * diff
    S = np.random.default_rng(14).standard_normal((6, r))
    lhs = np.sum(O.reconstruct(S, 5, 9, k) ** 2, axis=1)
    rhs = np.einsum("ia,ab,ib->i", S, M.astype(np.float64), S) / r
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes(monkeypatch):
    """Each mistake is planted in the oracle (on the CPU) and must fail a pin."""
    # 1) wrong sign scale 1/r: the Monte-Carlo mean is then G/r, far from G.
    d, k, r = 4, 64, 8
    G = np.random.default_rng(15).standard_normal((d, k))
    bad = lambda s, t, rr, kk: O.sign_matrix(s, t, rr, kk).astype(np.float64) / rr
    acc = np.zeros((d, k))
    for step in range(300):
        A = bad(1, step, r, k)
        acc += (G @ A.T) @ A
    err2 = np.sum((acc / 300 - G) ** 2)
    assert err2 / ((k - 1) * np.sum(G * G) / (r * 300)) > 2.0

    # 2) transposed sketch (S = dY^T X A^T computed as X^T dY ...): shape/values differ.
    n, d2, k2, r2 = 6, 5, 64, 4
    X, dY = _tiny(n, d2, k2, seed=16)
    A = O.projection_matrix(1, 0, r2, k2)
    good = (dY.T @ X) @ A.T
    wrong = dY.T @ (X @ A[::-1].T)           # row order of A flipped
    assert not np.allclose(good, wrong)

    # 3) v_old used in the denominator instead of v_new: the closed form fails.
    S = np.random.default_rng(17).standard_normal((3, 8))
    Gh = O.reconstruct(S, 0, 0, 64)
    m = np.mean(Gh ** 2, axis=1)
    dW_bad = -1e-3 * Gh / np.sqrt(0.0 + 1e-8)
    dW_good = -1e-3 * Gh / np.sqrt((1 - 0.999) * m + 1e-8)[:, None]
    assert not np.allclose(dW_bad, dW_good, rtol=1e-3)

    # 4) a dropped microbatch breaks linearity.
    mbs = [_tiny(9, 4, 64, seed=s) for s in (20, 21, 22)]
    S_all = O.sketch_accumulate(np.zeros((4, 8)), np.concatenate([m[0] for m in mbs]),
                                np.concatenate([m[1] for m in mbs]), 2, 2, 8)
    S_drop = np.zeros((4, 8))
    for X_, dY_ in mbs[:2]:
        S_drop = O.sketch_accumulate(S_drop, X_, dY_, 2, 2, 8)
    assert not np.allclose(S_all, S_drop, rtol=1e-6)

    # 5) a wrong finaliser shift breaks the published generator outputs.
    def bad_mix(z):
        z = np.array(z, dtype=np.uint64)
        with np.errstate(over="ignore"):
            z = (z ^ (z >> np.uint64(31))) * O._M1
            z = (z ^ (z >> np.uint64(27))) * O._M2
            return z ^ (z >> np.uint64(31))
    monkeypatch.setattr(O, "splitmix64_finalize", bad_mix)
    assert [int(x) for x in O.splitmix64_outputs(0, 2)] != _golden_words("splitmix64_seed0.txt")[:2]

    # 4) bias correction one step off (1 - beta2^(t+1)): the unit-rms first step fails.
    monkeypatch.setattr(O, "bias_corrected", lambda v, b, t: v / (1.0 - b ** (t + 1)) if t else v)
    S = np.random.default_rng(18).standard_normal((3, 8))
    _, _, _, dW = O.rowadam_apply(np.zeros((3, 64)), S, np.zeros(3), 0, 0, 0.9, 0.0, 1e-3, 1.0, t=1)
    assert not np.allclose(np.sum(dW * dW, axis=1), 1e-6 * 64, rtol=1e-6)
