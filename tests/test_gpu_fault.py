"""Failure detection on the GPU without a GPU fault.

A test hook makes one producer skip a pipeline stage, so the consumer's
bounded wait runs out: the kernel must record LOGRA_ERR_TIMEOUT in the device
status word, drain what it has in flight, free TMEM and return.  The context
stays usable: a clean call afterwards matches the oracle.
"""
import numpy as np
import pytest

from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

SHORT_WAIT = 4_000_000          # clock ticks (a few ms)
DEFAULT_WAIT = 2_000_000_000


@pytest.fixture(scope="module")
def L():
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    import rank_gradient_sketching_02_gb300 as L
    return L


def _clean_sketch(L):
    import torch
    n, d, k, r = 256, 264, 520, 64
    X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(77,))
    Xd, dYd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda()
    S = torch.zeros((d, r), dtype=torch.float32, device="cuda")
    L.logra_sketch_accumulate(Xd, dYd, S, 3, 4)
    torch.cuda.synchronize()
    want = O.sketch_accumulate(np.zeros((d, r)), Xd.double().cpu().numpy(), dYd.double().cpu().numpy(), 3, 4, r)
    got = S.double().cpu().numpy()
    return np.linalg.norm(got - want) / np.linalg.norm(want)


@pytest.mark.parametrize("r", [128, 256, 512])      # single-CTA accumulate; CTA-pair accumulate (256, 512)
def test_sketch_timeout_is_reported_and_context_survives(L, r):
    import torch
    assert L.logra_get_status() == 0
    L.logra_debug_inject(1, SHORT_WAIT)
    try:
        n, d, k = 512, 512, 1024
        X = torch.randn((n, k), device="cuda").to(torch.bfloat16)
        dY = torch.randn((n, d), device="cuda").to(torch.bfloat16)
        S = torch.zeros((d, r), device="cuda")
        L.logra_sketch_accumulate(X, dY, S, 1, 1)
        assert L.logra_get_status() == L.binding.LOGRA_ERR_TIMEOUT
    finally:
        L.logra_debug_inject(0, DEFAULT_WAIT)
    assert L.logra_get_status() == 0
    assert _clean_sketch(L) <= 1e-3


def test_apply_timeout_is_reported_and_context_survives(L):
    import torch
    d, k, r = 256, 512, 64
    S = torch.randn((d, r), device="cuda") * 1e-3
    L.logra_debug_inject(1, SHORT_WAIT)
    try:
        W = torch.zeros((d, k), device="cuda")
        v = torch.zeros(d, device="cuda")
        L.logra_rowadam_apply(W, S, v, 1, 1, 0.999, 1e-8, 1e-5, 1.0)
        assert L.logra_get_status() == L.binding.LOGRA_ERR_TIMEOUT
    finally:
        L.logra_debug_inject(0, DEFAULT_WAIT)
    W = torch.zeros((d, k), device="cuda")
    v = torch.zeros(d, device="cuda")
    L.logra_rowadam_apply(W, S, v, 1, 1, 0.999, 1e-8, 1e-5, 1.0)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    S64 = S.double().cpu().numpy()
    b2, eps, lr = (float(np.float32(x)) for x in (0.999, 1e-8, 1e-5))
    _, _, _, dW = O.rowadam_apply(np.zeros((d, k)), S64, np.zeros(d), 1, 1, b2, eps, lr, 1.0)
    got = W.double().cpu().numpy()
    assert np.linalg.norm(got - dW) / np.linalg.norm(dW) <= 1e-5


def test_dgrad_timeout_is_reported_and_context_survives(L):
    import torch
    n, d, k = 512, 512, 768
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    dY = torch.randn((n, d), generator=g, device="cuda").to(torch.bfloat16)
    W = torch.randn((d, k), generator=g, device="cuda").to(torch.bfloat16)
    dX = torch.zeros((n, k), dtype=torch.bfloat16, device="cuda")
    assert L.logra_get_status() == 0
    L.logra_debug_inject(1, SHORT_WAIT)
    try:
        L.logra_linear_backward(dY, W=W, dX=dX)
        assert L.logra_get_status() == L.binding.LOGRA_ERR_TIMEOUT
    finally:
        L.logra_debug_inject(0, DEFAULT_WAIT)
    assert L.logra_get_status() == 0
    L.logra_linear_backward(dY, W=W, dX=dX)
    torch.cuda.synchronize()
    assert L.logra_get_status() == 0
    want = O.input_gradient(dY.double().cpu().numpy(), W.double().cpu().numpy())
    got = dX.double().cpu().numpy()
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 2.0 ** -8
