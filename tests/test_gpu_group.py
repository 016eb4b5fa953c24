"""logra_rowadam_apply_group: several matrices per launch, against the oracle and
against one logra_rowadam_apply_ex call per matrix.

The grouped launches deal the work units of all matrices to one set of
persistent CTAs; every element of W, v, the bf16 copy and the sync sketch is
computed by the same arithmetic as in a single-matrix launch, so those are
compared bit for bit.  The norms are fp64 sums of per-CTA partials whose
partition depends on the grouping: relative 1e-12.
"""
import numpy as np
import pytest

from oracle import logra_oracle as O

pytestmark = pytest.mark.gpu

TOL_V, TOL_DW = 1e-5, 1e-5


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


def host64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _case(shapes, r, seed, w0_zero=True, norms_mask=None, lr=1e-5):
    """Host inputs of one group: per matrix S, v0, W0, seed, lr, c."""
    g = np.random.default_rng(seed)
    out = []
    for i, (d, k) in enumerate(shapes):
        S = (g.standard_normal((d, r)) * 1e-3 * np.exp(g.standard_normal((d, 1)))).astype(np.float32)
        v0 = (np.abs(g.standard_normal(d)) * 1e-8).astype(np.float32)
        W0 = np.zeros((d, k), np.float32) if w0_zero else (g.standard_normal((d, k)) * 0.02).astype(np.float32)
        out.append({"S": S, "v0": v0, "W0": W0, "seed": 1000 + 37 * i, "lr": float(np.float32(lr * (1 + i))),
                    "c": float(np.float32(0.5 + 0.25 * (i % 3))),
                    "norms": True if norms_mask is None else bool(norms_mask[i])})
    return out


def _device(case, torch):
    mats = []
    for m in case:
        d, k = m["W0"].shape
        r = m["S"].shape[1]
        mats.append({"W": torch.from_numpy(m["W0"]).cuda(), "S": torch.from_numpy(m["S"]).cuda(),
                     "v": torch.from_numpy(m["v0"]).cuda(), "seed": m["seed"], "lr": m["lr"], "c": m["c"],
                     "norms_out": torch.zeros(2, dtype=torch.float64, device="cuda") if m["norms"] else None,
                     "W_bf16_out": torch.empty((d, k), dtype=torch.bfloat16, device="cuda"),
                     "sync_sketch_out": torch.empty((d, r), dtype=torch.float32, device="cuda")})
    return mats


def _run_both(L, case, step, beta2, eps):
    import torch
    grouped, single = _device(case, torch), _device(case, torch)
    L.logra_rowadam_apply_group(grouped, step, beta2, eps)
    for m in single:
        L.logra_rowadam_apply_ex(m["W"], m["S"], m["v"], m["seed"], step, beta2, eps, m["lr"], m["c"],
                                 m["norms_out"], m["W_bf16_out"], m["sync_sketch_out"])
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    return grouped, single


# a decoder layer's seven projections, scaled down, with ragged row blocks and column tiles
LAYER = [(264, 520), (72, 520), (72, 520), (520, 264), (1032, 520), (1032, 520), (520, 1032)]


@pytest.mark.parametrize("r", [256, 64, 160])
def test_group_of_a_layer_against_oracle_and_single_calls(L, r):
    import torch
    beta2, eps = float(np.float32(0.999)), float(np.float32(1e-8))
    case = _case(LAYER, r, seed=r)
    grouped, single = _run_both(L, case, 5, beta2, eps)
    for m, g, s in zip(case, grouped, single):
        # bit for bit against the single-matrix call
        assert torch.equal(g["W"], s["W"])
        assert torch.equal(g["v"], s["v"])
        assert torch.equal(g["W_bf16_out"], s["W_bf16_out"])
        assert torch.equal(g["sync_sketch_out"], s["sync_sketch_out"])
        ng, ns = g["norms_out"].cpu().numpy(), s["norms_out"].cpu().numpy()
        assert np.all(np.abs(ng - ns) <= 1e-12 * np.abs(ns))
        # and against the oracle (W0 = 0, so W = dW)
        _, v_or, n_or, dW_or = O.rowadam_apply(m["W0"].astype(np.float64), m["S"].astype(np.float64),
                                               m["v0"].astype(np.float64), m["seed"], 5, beta2, eps, m["lr"],
                                               m["c"])
        assert rel(host64(g["v"]), v_or) <= TOL_V
        assert rel(host64(g["W"]), dW_or) <= TOL_DW
        assert abs(ng[0] - n_or[0]) <= TOL_V * n_or[0]
        assert abs(ng[1] - n_or[1]) <= TOL_V * n_or[1]
        assert torch.equal(g["W_bf16_out"], g["W"].to(torch.bfloat16))
        assert rel(host64(g["sync_sketch_out"]), O.sync_sketch(m["S"], v_or, eps, m["lr"], m["c"])) <= TOL_V


def test_group_spanning_two_launch_groups_with_optional_outputs(L):
    """Ten matrices (launch groups of 8 and 2), realistic W0, some without norms."""
    import torch
    beta2, eps = float(np.float32(0.99)), float(np.float32(1e-8))
    shapes = [(136, 264), (8, 8), (128, 256), (392, 72), (40, 1000), (264, 136), (16, 520), (520, 16),
              (200, 344), (64, 64)]
    # lr large enough that dW stands well above the fp32 rounding of W0 + dW (ulp(0.02) ~ 2e-9)
    case = _case(shapes, 96, seed=3, w0_zero=False, norms_mask=[1, 0, 1, 1, 0, 1, 1, 1, 0, 1], lr=1e-4)
    grouped, single = _run_both(L, case, 2, beta2, eps)
    for m, g, s in zip(case, grouped, single):
        assert torch.equal(g["W"], s["W"])
        assert torch.equal(g["v"], s["v"])
        assert torch.equal(g["W_bf16_out"], s["W_bf16_out"])
        assert torch.equal(g["sync_sketch_out"], s["sync_sketch_out"])
        if m["norms"]:
            ng, ns = g["norms_out"].cpu().numpy(), s["norms_out"].cpu().numpy()
            assert np.all(np.abs(ng - ns) <= 1e-12 * np.abs(ns))
        _, v_or, n_or, dW_or = O.rowadam_apply(m["W0"].astype(np.float64), m["S"].astype(np.float64),
                                               m["v0"].astype(np.float64), m["seed"], 2, beta2, eps, m["lr"],
                                               m["c"])
        assert rel(host64(g["v"]), v_or) <= TOL_V
        assert rel(host64(g["W"]) - m["W0"].astype(np.float64), dW_or) <= TOL_DW
        if m["norms"]:
            assert abs(g["norms_out"].cpu().numpy()[1] - n_or[1]) <= TOL_V * n_or[1]


def test_group_of_one_and_empty(L):
    import torch
    beta2, eps = float(np.float32(0.999)), float(np.float32(1e-8))
    case = _case([(256, 512)], 32, seed=9)
    grouped, single = _run_both(L, case, 0, beta2, eps)
    assert torch.equal(grouped[0]["W"], single[0]["W"])
    assert torch.equal(grouped[0]["norms_out"], single[0]["norms_out"])   # same partition: same sums
    L.logra_rowadam_apply_group([], 0, beta2, eps)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0


def test_group_7b_layer_fullsize(L):
    """The seven projections of a 7B-class layer (q/o 3584x3584, k/v 512x3584, gate/up 18944x3584,
    down 3584x18944; r = 256) in one grouped call, as the bench issues them: bit for bit against
    one call per matrix, and sampled rows against the oracle's row-wise RowAdam."""
    import torch
    from rank_gradient_sketching_02_gb300 import synth
    r = 256
    shapes = [(3584, 3584), (512, 3584), (512, 3584), (3584, 3584), (18944, 3584), (18944, 3584), (3584, 18944)]
    # lr large enough that dW (~3e-3) stands well above the fp32 rounding of W0 + dW (ulp(0.02) ~ 2e-9)
    beta2, eps, lr = (float(np.float32(x)) for x in (synth.BETA2, synth.EPS, 1e-4))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    grouped, single, host = [], [], []
    for i, (d, k) in enumerate(shapes):
        S = torch.randn((d, r), device="cuda", generator=gen) * 1e-3
        v0 = torch.rand(d, device="cuda", generator=gen) * 1e-9
        W0 = torch.randn((d, k), device="cuda", generator=gen) * 0.02
        for dst in (grouped, single):
            dst.append({"W": W0.clone(), "S": S, "v": v0.clone(), "seed": synth.matrix_seed(2026, 0, i), "lr": lr,
                        "c": 1.0, "norms_out": torch.zeros(2, dtype=torch.float64, device="cuda"),
                        "W_bf16_out": torch.empty((d, k), dtype=torch.bfloat16, device="cuda")})
        host.append((S.double().cpu().numpy(), v0.double().cpu().numpy(), W0))
    L.logra_rowadam_apply_group(grouped, 3, beta2, eps)
    for m in single:
        L.logra_rowadam_apply_ex(m["W"], m["S"], m["v"], m["seed"], 3, beta2, eps, m["lr"], m["c"],
                                 m["norms_out"], m["W_bf16_out"], None)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    for i, ((d, k), g, s, (Sh, vh, W0)) in enumerate(zip(shapes, grouped, single, host)):
        assert torch.equal(g["W"], s["W"]), i
        assert torch.equal(g["v"], s["v"]), i
        assert torch.equal(g["W_bf16_out"], s["W_bf16_out"]), i
        ng, ns = g["norms_out"].cpu().numpy(), s["norms_out"].cpu().numpy()
        assert np.all(np.abs(ng - ns) <= 1e-12 * np.abs(ns)), i
        rows = np.random.default_rng(i).choice(d, size=4, replace=False)
        v_or, dW_or, _ = O.rowadam_rows(Sh[rows], vh[rows], k, g["seed"], 3, beta2, eps, lr, 1.0)
        assert rel(g["v"].double().cpu().numpy()[rows], v_or) <= TOL_V
        idx = torch.from_numpy(rows).cuda()
        dW = (g["W"][idx].double() - W0[idx].double()).cpu().numpy()
        assert rel(dW, dW_or) <= TOL_DW


def test_group_with_bias_correction_per_matrix(L):
    """Items with different t (0 = uncorrected) against one logra_rowadam_apply_bc call each."""
    import torch
    beta2, eps = float(np.float32(0.99)), float(np.float32(1e-8))
    shapes = [(264, 520), (72, 520), (520, 264)]
    ts = [0, 1, 7]
    case = _case(shapes, 128, seed=11)
    grouped, single = _device(case, torch), _device(case, torch)
    for m, t in zip(grouped, ts):
        m["t"] = t
    L.logra_rowadam_apply_group(grouped, 4, beta2, eps)
    for m, t in zip(single, ts):
        L.logra_rowadam_apply_bc(m["W"], m["S"], m["v"], m["seed"], 4, beta2, eps, m["lr"], m["c"], t,
                                 m["norms_out"], m["W_bf16_out"], m["sync_sketch_out"])
    torch.cuda.synchronize()
    for m, g, s, t in zip(case, grouped, single, ts):
        assert torch.equal(g["W"], s["W"]) and torch.equal(g["v"], s["v"])
        assert torch.equal(g["sync_sketch_out"], s["sync_sketch_out"])
        _, v_or, _, dW_or = O.rowadam_apply(m["W0"].astype(np.float64), m["S"].astype(np.float64),
                                            m["v0"].astype(np.float64), m["seed"], 4, beta2, eps, m["lr"], m["c"],
                                            t=t)
        assert rel(host64(g["W"]), dW_or) <= TOL_DW
