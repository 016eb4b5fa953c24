"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (relative Frobenius unless stated):
  * A                         bit-exact
  * S, bf16 inputs            1e-3   (fp32 accumulation of exact bf16 products)
  * S, fp32 inputs            1e-5
  * v, norms                  1e-5   (apply checked stage-wise on the kernel's own S)
  * dW (W0 = 0, so W = dW)    1e-5
  * W with a realistic W0     W_new - W_old vs dW_oracle 1e-5 (Frobenius), and elementwise
                              |W - fl32(W0 + dW_oracle)| <= 2 ulp(W) + 1e-4 rms_row(dW)
"""
import math

import numpy as np
import pytest

from canary import Guarded
from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_S_BF16, TOL_S_F32, TOL_V, TOL_DW = 1e-3, 1e-5, 1e-5, 1e-5


@pytest.fixture(scope="module")
def L():
    import torch
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    torch.cuda.init()
    return L


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def to_dev(a, dtype):
    import torch
    if dtype == "bf16":
        return synth.to_bf16_bits(a).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


# ------------------------------------------------------------------ sign matrix
@pytest.mark.parametrize("seed,step,r,k", [(0, 0, 32, 512), (12345, 7, 256, 1536), (2**63 + 5, 2**40, 512, 200),
                                           (3, 1, 64, 1), (9, 9, 128, 27648)])
def test_sign_matrix_bit_exact(L, seed, step, r, k):
    import torch
    gA = Guarded((r, k), torch.float32)
    L.logra_sign_matrix(seed, step, r, k, gA.t)
    gA.check("A")
    A = gA.t.cpu().numpy()
    want = O.projection_matrix_fp32(seed, step, r, k)
    assert np.array_equal(A.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------------ sketch
def run_sketch(L, mbs, d, r, dtype, seed, step):
    import torch
    gS = Guarded((d, r), torch.float32, fill=0.0)           # S between guard regions
    S = gS.t
    S_or = np.zeros((d, r))
    for X, dY in mbs:
        Xd, dYd = to_dev(X, dtype), to_dev(dY, dtype)
        L.logra_sketch_accumulate(Xd, dYd, S, seed, step)
        S_or = O.sketch_accumulate(S_or, host64(Xd), host64(dYd), seed, step, r)
    gS.check("S")
    return host64(S), S_or


def test_sketch_tiny_fp32(L):
    w = synth.WORKLOADS["tiny"]
    (_, d, k), = w.matrices
    mbs = [synth.host_microbatch(w.tokens, d, k, dy_kind=w.dy_kind, dy_std=w.dy_std, mask_frac=w.mask_frac,
                                 key=(0, 0, 0, mb))[:2] for mb in range(w.microbatches)]
    S, S_or = run_sketch(L, mbs, d, w.r, "f32", 0, 0)
    assert rel(S, S_or) <= TOL_S_F32


@pytest.mark.parametrize("n,d,k,r", [(4096, 1536, 1536, 256), (300, 264, 520, 96), (1, 8, 8, 32),
                                     (777, 1024, 200, 512), (129, 4104, 136, 128), (640, 392, 1032, 384)])
def test_sketch_bf16(L, n, d, k, r):
    mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(1, n, d, k, r, mb))[:2]
           for mb in range(2)]
    S, S_or = run_sketch(L, mbs, d, r, "bf16", 77, 3)
    assert rel(S, S_or) <= TOL_S_BF16


def test_sketch_scratch_reuse_across_shapes(L):
    """Calls on one stream whose P^T scratch shrinks, grows and comes back, with an apply and
    an fp32 sketch (both overwrite the scratch) in between: each call's accumulate leaves its
    P^T at zero for the next projection, and the library memsets only what it cannot vouch for."""
    import torch
    seq = [(1024, 264, 1032, 128, "bf16"), (300, 72, 520, 256, "bf16"), (2048, 136, 2056, 256, "bf16"),
           ("apply",), (1024, 264, 1032, 128, "bf16"), (257, 64, 72, 32, "f32"), (2048, 136, 2056, 256, "bf16"),
           (2048, 136, 2056, 256, "bf16")]
    for i, job in enumerate(seq):
        if job[0] == "apply":
            W = torch.zeros((256, 512), device="cuda")
            L.logra_rowadam_apply(W, to_dev(_sketch_like(256, 32, 3), "f32"), torch.zeros(256, device="cuda"),
                                  1, 1, 0.999, 1e-8, 1e-5, 1.0)
            continue
        n, d, k, r, dt = job
        mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(6, i, mb))[:2]
               for mb in range(2)]
        S, S_or = run_sketch(L, mbs, d, r, dt, 40 + i, i)
        assert rel(S, S_or) <= (TOL_S_BF16 if dt == "bf16" else TOL_S_F32), i


@pytest.mark.parametrize("n,d,k,r", [(257, 64, 72, 32), (100, 24, 1000, 64)])
def test_sketch_fp32_ragged(L, n, d, k, r):
    mbs = [synth.host_microbatch(n, d, k, dy_kind="gauss", dy_std=1e-3, mask_frac=0.2, key=(2, n, mb))[:2]
           for mb in range(3)]
    S, S_or = run_sketch(L, mbs, d, r, "f32", 5, 2)
    assert rel(S, S_or) <= TOL_S_F32


@pytest.mark.parametrize("n,d,k,r", [(777, 1032, 520, 256), (300, 264, 1032, 512), (129, 4104, 136, 128),
                                     (1000, 1536, 1536, 384)])
def test_sketch_fp32_tensor_core_shapes(L, n, d, k, r):
    """fp32 inputs through the stacked bf16 planes on both accumulate kernels (CTA pairs at
    r = 256 and 512, one CTA otherwise), with the lognormal gradient scales: dropping the
    second plane of X or dY would leave an error near 1e-3, a hundred times the bound."""
    mbs = [synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(8, n, d, k, r, mb))[:2]
           for mb in range(2)]
    S, S_or = run_sketch(L, mbs, d, r, "f32", 11, 4)
    assert rel(S, S_or) <= TOL_S_F32


def test_sketch_n0_is_noop_and_padding_rows(L):
    import torch
    d, k, r = 64, 128, 32
    S = torch.ones((d, r), dtype=torch.float32, device="cuda")
    X = torch.zeros((0, k), dtype=torch.bfloat16, device="cuda")
    dY = torch.zeros((0, d), dtype=torch.bfloat16, device="cuda")
    L.logra_sketch_accumulate(X, dY, S, 1, 1)
    X = torch.zeros((50, k), dtype=torch.bfloat16, device="cuda")
    dY = torch.randn((50, d), device="cuda").to(torch.bfloat16)
    L.logra_sketch_accumulate(X, dY, S, 1, 1)              # all-padding X: S unchanged
    torch.cuda.synchronize()
    assert torch.equal(S, torch.ones_like(S))


def test_sketch_rejects_bad_shapes(L):
    import torch
    S = torch.zeros((12, 32), device="cuda")
    X = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    dY = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.LograError):
        L.logra_sketch_accumulate(X, dY, S, 0, 0)
    S = torch.zeros((16, 40), device="cuda")
    dY = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.LograError):
        L.logra_sketch_accumulate(X, dY, S, 0, 0)


# ------------------------------------------------------------------ RowAdam apply
def _sketch_like(d, r, seed, scale=1e-3):
    g = np.random.default_rng(seed)
    return (g.standard_normal((d, r)) * scale * np.exp(g.standard_normal((d, 1)))).astype(np.float32)


@pytest.mark.parametrize("d,k,r", [(256, 512, 32), (1536, 1536, 256), (40, 1000, 64), (520, 264, 512),
                                   (8, 8, 32), (392, 1032, 384), (136, 2056, 96), (264, 72, 160),
                                   (40, 4104, 64), (24, 8200, 32)])   # Gram words over 2 and 3 blocks
def test_apply_stagewise_zero_w0(L, d, k, r):
    import torch
    S32 = _sketch_like(d, r, d + k)
    v0 = (np.abs(np.random.default_rng(1).standard_normal(d)) * 1e-8).astype(np.float32)
    S = to_dev(S32, "f32")
    guards = [Guarded((d,), torch.float32, fill=to_dev(v0, "f32")), Guarded((d, k), torch.float32, fill=0.0),
              Guarded((d, k), torch.bfloat16), Guarded((d, r), torch.float32), Guarded((2,), torch.float64, fill=0.0)]
    v, W, Wb, sync, norms = (g.t for g in guards)
    beta2, eps, lr, c = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-5, 0.75))
    L.logra_rowadam_apply_ex(W, S, v, 11, 4, beta2, eps, lr, c, norms, Wb, sync)
    for g, what in zip(guards, ("v", "W", "W bf16", "sync sketch", "norms")):
        g.check(what)
    W_or, v_or, n_or, dW_or = O.rowadam_apply(np.zeros((d, k)), S32.astype(np.float64), v0.astype(np.float64),
                                              11, 4, beta2, eps, lr, c)
    assert rel(host64(v), v_or) <= TOL_V
    assert rel(host64(W), dW_or) <= TOL_DW
    nr = norms.cpu().numpy()
    assert abs(nr[0] - n_or[0]) <= TOL_V * n_or[0]
    assert abs(nr[1] - n_or[1]) <= TOL_V * n_or[1]
    assert torch.equal(Wb, W.to(torch.bfloat16))                       # RN-even copy of the master
    assert rel(host64(sync), O.sync_sketch(S32, v_or, eps, lr, c)) <= TOL_V


def test_apply_realistic_w0_and_two_steps(L):
    import torch
    d, k, r = 264, 776, 128
    W0 = synth.host_weight(d, k, key=(3,))
    W = to_dev(W0, "f32")
    v = torch.zeros(d, dtype=torch.float32, device="cuda")
    W_or, v_or = W0.astype(np.float64), np.zeros(d)
    beta2, eps, lr, c = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-4, 1.0))
    for step in range(2):
        S32 = _sketch_like(d, r, 100 + step)
        v_before = host64(v)
        Wprev = host64(W)
        L.logra_rowadam_apply(W, to_dev(S32, "f32"), v, 21, step, beta2, eps, lr, c)
        torch.cuda.synchronize()
        _, v_or, _, dW = O.rowadam_apply(Wprev, S32.astype(np.float64), v_before, 21, step, beta2, eps, lr, c)
        assert rel(host64(v), v_or) <= TOL_V
        Wg = host64(W)
        want = (Wprev + dW).astype(np.float32).astype(np.float64)
        ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
        # the applied update (W_new - W_old) against the oracle's dW, Frobenius;
        # it includes the fp32 rounding of W_new, ~ulp(W)/2 per element
        assert rel(Wg - Wprev, dW) <= TOL_DW
        # elementwise sanity: an fp32 sum of r signed terms loses relative
        # accuracy where a row's terms cancel, so bound by the row's scale
        row_rms = np.sqrt(np.mean(dW * dW, axis=1, keepdims=True))
        assert np.all(np.abs(Wg - want) <= 2.01 * ulp + 1e-4 * row_rms)


def test_apply_zero_sketch_and_zero_scale(L):
    import torch
    d, k, r = 64, 256, 32
    W0 = synth.host_weight(d, k, key=(4,))
    W = to_dev(W0, "f32")
    v0 = np.full(d, 2e-9, dtype=np.float32)
    v = to_dev(v0, "f32")
    norms = torch.zeros(2, dtype=torch.float64, device="cuda")
    L.logra_rowadam_apply(W, torch.zeros((d, r), device="cuda"), v, 0, 0, 0.9, 1e-8, 1e-3, 1.0, norms)
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy(), W0)
    np.testing.assert_allclose(v.cpu().numpy(), np.float32(0.9) * v0, rtol=1e-6)
    assert norms.cpu().tolist() == [0.0, 0.0]
    S32 = _sketch_like(d, r, 5)
    L.logra_rowadam_apply(W, to_dev(S32, "f32"), v, 0, 0, 0.9, 1e-8, 1e-3, 0.0, norms)   # c = 0
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy(), W0)
    assert norms.cpu().numpy()[1] == 0.0


def test_predict_matches_apply_norms_and_writes_nothing(L):
    import torch
    d, k, r = 128, 512, 64
    S32 = _sketch_like(d, r, 6)
    v0 = np.full(d, 1e-9, dtype=np.float32)
    S, v = to_dev(S32, "f32"), to_dev(v0, "f32")
    norms = torch.zeros(2, dtype=torch.float64, device="cuda")
    L.logra_rowadam_predict(S, v, k, 8, 8, 0.999, 1e-8, 1e-5, norms)
    torch.cuda.synchronize()
    assert np.array_equal(v.cpu().numpy(), v0)
    _, _, n_or, _ = O.rowadam_apply(np.zeros((d, k)), S32.astype(np.float64), v0.astype(np.float64), 8, 8,
                                    float(np.float32(0.999)), float(np.float32(1e-8)), float(np.float32(1e-5)), 1.0)
    nr = norms.cpu().numpy()
    assert abs(nr[0] - n_or[0]) <= TOL_V * n_or[0] and abs(nr[1] - n_or[1]) <= TOL_V * n_or[1]


# ------------------------------------------------------------------ reconstruct
@pytest.mark.parametrize("d,k,r", [(256, 512, 32), (72, 1544, 256), (16, 8, 512)])
def test_reconstruct(L, d, k, r):
    import torch
    S32 = _sketch_like(d, r, 7)
    S = to_dev(S32, "f32")
    want = O.reconstruct(S32.astype(np.float64), 13, 2, k)
    gout = Guarded((d, k), torch.float32)
    out = gout.t
    L.logra_reconstruct(S, k, 13, 2, out)
    gout.check("reconstruct out")
    assert rel(host64(out), want) <= 1e-5
    base = np.random.default_rng(8).standard_normal((d, k)).astype(np.float32)
    out = to_dev(base, "f32")
    L.logra_reconstruct(S, k, 13, 2, out, accumulate=True)
    torch.cuda.synchronize()
    assert rel(host64(out) - base, want) <= 1e-4
    gob = Guarded((d, k), torch.bfloat16)
    ob = gob.t
    L.logra_reconstruct(S, k, 13, 2, ob)
    gob.check("reconstruct bf16 out")
    assert rel(host64(ob), want) <= 4e-3          # one bf16 rounding of each element


def test_sync_sketch_rebuilds_applied_update(L):
    import torch
    d, k, r = 128, 384, 64
    S32 = _sketch_like(d, r, 9)
    S = to_dev(S32, "f32")
    v = torch.zeros(d, device="cuda")
    W = torch.zeros((d, k), device="cuda")
    sync = torch.empty((d, r), device="cuda")
    L.logra_rowadam_apply_ex(W, S, v, 1, 1, 0.999, 1e-8, 1e-5, 1.0, None, None, sync)
    rebuilt = torch.zeros((d, k), device="cuda")
    L.logra_reconstruct(sync, k, 1, 1, rebuilt, accumulate=True)
    torch.cuda.synchronize()
    assert rel(host64(rebuilt), host64(W)) <= 1e-5


def test_status_word_clean(L):
    assert L.logra_get_status() == 0


# ------------------------------------------------------------------ bias-corrected variant
@pytest.mark.parametrize("t", [1, 3])
def test_apply_bias_corrected(L, t):
    import torch
    d, k, r = 392, 1032, 128
    S32 = _sketch_like(d, r, 50 + t)
    v0 = (np.abs(np.random.default_rng(t).standard_normal(d)) * 1e-8).astype(np.float32)
    S, v = to_dev(S32, "f32"), to_dev(v0, "f32")
    W = torch.zeros((d, k), dtype=torch.float32, device="cuda")
    sync = torch.empty((d, r), dtype=torch.float32, device="cuda")
    norms = torch.zeros(2, dtype=torch.float64, device="cuda")
    pred = torch.zeros(2, dtype=torch.float64, device="cuda")
    beta2, eps, lr, c = (float(np.float32(x)) for x in (0.99, 1e-8, 1e-5, 0.8))
    L.logra_rowadam_predict_bc(S, v, k, 3, t, beta2, eps, lr, t, pred)
    L.logra_rowadam_apply_bc(W, S, v, 3, t, beta2, eps, lr, c, t, norms, None, sync)
    torch.cuda.synchronize()
    _, v_or, n_or, dW_or = O.rowadam_apply(np.zeros((d, k)), S32.astype(np.float64), v0.astype(np.float64), 3, t,
                                           beta2, eps, lr, c, t=t)
    assert rel(host64(v), v_or) <= TOL_V                     # the stored v is uncorrected
    assert rel(host64(W), dW_or) <= TOL_DW
    nr = norms.cpu().numpy()
    assert abs(nr[0] - n_or[0]) <= TOL_V * n_or[0] and abs(nr[1] - n_or[1]) <= TOL_V * n_or[1]
    pr = pred.cpu().numpy()                                   # predict at c = 1: c^2 scaling
    assert abs(pr[1] * c * c - nr[1]) <= 1e-6 * nr[1]
    assert rel(host64(sync), O.sync_sketch(S32, v_or, eps, lr, c, beta2=beta2, t=t)) <= TOL_V


def test_apply_bias_correction_t0_is_the_plain_apply(L):
    import torch
    d, k, r = 136, 520, 64
    S = to_dev(_sketch_like(d, r, 60), "f32")
    outs = []
    for fn in ("plain", "bc0"):
        v = torch.full((d,), 1e-9, device="cuda")
        W = torch.zeros((d, k), device="cuda")
        norms = torch.zeros(2, dtype=torch.float64, device="cuda")
        if fn == "plain":
            L.logra_rowadam_apply_ex(W, S, v, 5, 5, 0.999, 1e-8, 1e-5, 1.0, norms)
        else:
            L.logra_rowadam_apply_bc(W, S, v, 5, 5, 0.999, 1e-8, 1e-5, 1.0, 0, norms)
        outs.append((W, v, norms))
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
