"""logra_linear_backward through the C ABI: dX = dY W and the sketch, against the fp64 oracle.

dX tolerance, derived from the arithmetic (the pages fix none for the input
gradient, which the method leaves as it is): the kernel adds the exact
products of bf16 operands in fp32 and rounds the sum once to bf16.  Every
element therefore lies within one bf16 ulp of the exact sum plus the fp32
summation error, bounded by d * 2^-24 * sum_a |dY_ta W_aj|; on random data
nearly all elements (>= 97% asked) equal the exact sum rounded to bf16, and the relative
Frobenius error stays below 2^-8 (half a bf16 ulp at the bottom of a binade).
S is checked as the sketch always is (relative Frobenius 1e-3 for bf16 inputs).
"""
import numpy as np
import pytest

from canary import Guarded
from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_S_BF16 = 1e-3
TOL_DX_FROB = 2.0 ** -8


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
    return np.linalg.norm(np.asarray(a, np.float64) - b) / (nb if nb > 0 else 1.0)


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)


def round_bf16(x):
    import torch
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def check_dx(got, dY64, W64, exact_frac=0.97):
    want = O.input_gradient(dY64, W64)
    absum = np.abs(dY64) @ np.abs(W64)
    d = dY64.shape[1]
    bound = bf16_ulp(want) + d * 2.0 ** -24 * absum
    err = np.abs(got - want)
    assert np.all(err <= bound), f"max excess {np.max(err - bound)} at {np.unravel_index(np.argmax(err - bound), err.shape)}"
    if want.size >= 1000:
        same = np.mean(got == round_bf16(want))
        assert same >= exact_frac, same
    assert rel(got, want) <= TOL_DX_FROB


def host64(t):
    return t.detach().double().cpu().numpy()


# ------------------------------------------------------------------ one-hot rows: bit-exact layout check
@pytest.mark.parametrize("n,d,k", [(256, 64, 256), (300, 200, 136), (77, 8, 8), (1000, 776, 520), (513, 4104, 1032),
                                   (256, 512, 3584)])
def test_dgrad_one_hot_rows_pick_rows_of_w_exactly(L, n, d, k):
    """dY row t = e_{a_t}: dX row t is row a_t of W, bit for bit (one exact product per sum;
    the other terms are signed zeros, so a -0 of W comes out as +0, the IEEE sum)."""
    import torch
    g = np.random.default_rng(n * 7 + d)
    a = g.integers(0, d, n)
    dY = torch.zeros((n, d), dtype=torch.bfloat16)
    dY[torch.arange(n), torch.from_numpy(a)] = 1.0
    W = synth.to_bf16_bits(g.standard_normal((d, k), dtype=np.float32))
    gX = Guarded((n, k), torch.bfloat16, fill=float("nan"))
    L.logra_linear_backward(dY.cuda(), W=W.cuda(), dX=gX.t)
    gX.check("dX")
    got = gX.t.cpu()
    want = W[torch.from_numpy(a)]
    same = (got.view(torch.int16) == want.view(torch.int16)) | ((got == 0) & (want == 0))
    assert bool(same.all()), int((~same).sum())


# ------------------------------------------------------------------ random inputs vs the oracle
@pytest.mark.parametrize("n,d,k", [(256, 256, 256), (300, 200, 136), (1000, 776, 520), (2048, 1032, 4104),
                                   (4096, 3584, 512), (520, 18944, 264)])
def test_dgrad_matches_oracle(L, n, d, k):
    import torch
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="gauss", key=(n, d, k))
    W = synth.host_weight(d, k, std=0.02, key=(d, k))
    dYd, Wd = synth.to_bf16_bits(dY).cuda(), synth.to_bf16_bits(W).cuda()
    gX = Guarded((n, k), torch.bfloat16, fill=float("nan"))
    L.logra_linear_backward(dYd, W=Wd, dX=gX.t)
    gX.check("dX")
    check_dx(host64(gX.t), host64(dYd), host64(Wd))


@pytest.mark.parametrize("n,d,k,r,mask", [(512, 264, 520, 64, 0.25), (1000, 776, 1032, 256, 0.0),
                                          (2048, 1536, 1536, 512, 0.1), (300, 136, 200, 32, 0.0)])
def test_linear_backward_gives_dx_and_sketch(L, n, d, k, r, mask):
    """One call: dX as the oracle's input gradient, S as the oracle's sketch (on a nonzero S)."""
    import torch
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=mask, key=(5, n, d))
    W = synth.host_weight(d, k, std=0.02, key=(6, d, k))
    Xd, dYd, Wd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda(), synth.to_bf16_bits(W).cuda()
    S0 = np.random.default_rng(9).standard_normal((d, r)).astype(np.float32) * np.float32(1e-3)
    gS = Guarded((d, r), torch.float32, fill=torch.from_numpy(S0))
    gX = Guarded((n, k), torch.bfloat16, fill=float("nan"))
    seed, step = 1234 + n, 7
    L.logra_linear_backward(dYd, W=Wd, dX=gX.t, X=Xd, S=gS.t, seed=seed, step=step)
    gS.check("S")
    gX.check("dX")
    dX_want, S_want = O.linear_backward(S0.astype(np.float64), host64(Xd), host64(dYd), host64(Wd), seed, step, r)
    check_dx(host64(gX.t), host64(dYd), host64(Wd))
    assert rel(host64(gS.t) - S0, S_want - S0) <= TOL_S_BF16


def test_sketch_only_and_dx_only_forms(L):
    import torch
    n, d, k, r = 640, 392, 776, 128
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="gauss", key=(17,))
    W = synth.host_weight(d, k, key=(18,))
    Xd, dYd, Wd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda(), synth.to_bf16_bits(W).cuda()
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    L.logra_linear_backward(dYd, X=Xd, S=S, seed=3, step=4)
    want = O.sketch_accumulate(np.zeros((d, r)), host64(Xd), host64(dYd), 3, 4, r)
    assert rel(host64(S), want) <= TOL_S_BF16
    dX = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    L.logra_linear_backward(dYd, W=Wd, dX=dX)
    check_dx(host64(dX), host64(dYd), host64(Wd))


# ------------------------------------------------------------------ full size: 7B gate projection, sampled rows
def test_dgrad_full_size_gate_sampled_rows(L):
    """n = 8192 tokens, d = 18944, k = 3584 (the 7B-class MLP gate): 48 rows of dX vs the oracle."""
    import torch
    n, d, k = 8192, 18944, 3584
    g = torch.Generator(device="cuda")
    g.manual_seed(42)
    dY = torch.randn((n, d), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((d, k), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    gX = Guarded((n, k), torch.bfloat16, fill=float("nan"))
    L.logra_linear_backward(dY, W=W, dX=gX.t)
    gX.check("dX")
    assert L.logra_get_status() == 0
    rows = np.sort(np.random.default_rng(43).choice(n, 48, replace=False))
    rows[-1] = n - 1
    rows_t = torch.from_numpy(rows).cuda()
    check_dx(host64(gX.t[rows_t]), host64(dY[rows_t]), host64(W))
    assert not torch.isnan(gX.t.float()).any()


# ------------------------------------------------------------------ scheduling: graphs, streams, late pairs
def test_linear_backward_replayed_as_cuda_graph(L):
    """Captured once (the first eager call allocates the stream's counters and workspace), replayed:
    every replay gives the oracle's dX and sketch, and the tile counter is left at zero each time."""
    import torch
    n, d, k, r = 1024, 1032, 776, 128
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="gauss", key=(31,))
    W = synth.host_weight(d, k, key=(32,))
    Xd, dYd, Wd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda(), synth.to_bf16_bits(W).cuda()
    s = torch.cuda.Stream()
    dX = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        L.logra_linear_backward(dYd, W=Wd, dX=dX, X=Xd, S=S, seed=5, step=6)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        S.zero_()
        dX.zero_()
        L.logra_linear_backward(dYd, W=Wd, dX=dX, X=Xd, S=S, seed=5, step=6)
    want_S = O.sketch_accumulate(np.zeros((d, r)), host64(Xd), host64(dYd), 5, 6, r)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        check_dx(host64(dX), host64(dYd), host64(Wd))
        assert rel(host64(S), want_S) <= TOL_S_BF16
    assert L.logra_get_status() == 0


def test_dgrad_on_concurrent_streams_with_late_pairs(L):
    """Two dX calls on two streams at once (each stream has its own tile counter) while a third
    stream keeps SMs busy with sketches, so that some CTA pairs start late and take fewer tiles."""
    import torch
    shapes = [(2048, 3584, 1032), (1536, 2056, 3584)]
    ins, outs = [], []
    for i, (n, d, k) in enumerate(shapes):
        _, dY, _ = synth.host_microbatch(n, d, 8, dy_kind="gauss", key=(40 + i,))
        W = synth.host_weight(d, k, key=(50 + i,))
        ins.append((synth.to_bf16_bits(dY).cuda(), synth.to_bf16_bits(W).cuda()))
        outs.append(torch.empty((n, k), dtype=torch.bfloat16, device="cuda"))
    Xb = torch.randn((8192, 3584), device="cuda").to(torch.bfloat16)
    dYb = torch.randn((8192, 4096), device="cuda").to(torch.bfloat16)
    Sb = torch.zeros((4096, 256), device="cuda")
    streams = [torch.cuda.Stream() for _ in range(3)]
    torch.cuda.synchronize()
    for rep in range(3):
        with torch.cuda.stream(streams[2]):
            for _ in range(4):
                L.logra_sketch_accumulate(Xb, dYb, Sb, 1, rep)
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs[i].fill_(float("nan"))
                L.logra_linear_backward(ins[i][0], W=ins[i][1], dX=outs[i])
        torch.cuda.synchronize()
        for i in range(2):
            check_dx(host64(outs[i]), host64(ins[i][0]), host64(ins[i][1]))
    assert L.logra_get_status() == 0
