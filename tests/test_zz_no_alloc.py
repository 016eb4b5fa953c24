"""The allocation-free sketch entry point against the regular one.

Callers that may not allocate device memory (a framework whose caching
allocator owns all device memory, a real-time loop that must not block in the
driver, a runtime whose device memory is fixed at start-up) use
logra_sketch_accumulate_noalloc, whose scratch is a fixed device array inside
the library.  Its results must match logra_sketch_accumulate's on the same
inputs, call after call (the shared scratch keeps the previous call's bytes).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

from rank_gradient_sketching_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_S = 1e-3   # the sketch tolerance of the parity tests (bf16 inputs)


@pytest.fixture(scope="module")
def lib():
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    from rank_gradient_sketching_02_gb300 import binding
    h = binding.lib()
    f = h.logra_sketch_accumulate_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
    return h


def test_noalloc_matches_regular_entry_point_twice(lib):
    import torch
    from rank_gradient_sketching_02_gb300 import binding
    stream = torch.cuda.current_stream().cuda_stream
    for call, (n, d, k, r) in enumerate([(1000, 1544, 776, 256), (4096, 512, 1536, 128)]):
        X, dY, _ = synth.host_microbatch(n, d, k, dy_kind="lognormal", mask_frac=0.25, key=(31, call))
        Xd, dYd = synth.to_bf16_bits(X).cuda(), synth.to_bf16_bits(dY).cuda()
        S_ref = torch.full((d, r), 0.5, dtype=torch.float32, device="cuda")
        S_new = S_ref.clone()
        st = lib.logra_sketch_accumulate(Xd.data_ptr(), dYd.data_ptr(), binding.LOGRA_BF16, n, d, k, r, 5, call,
                                         S_ref.data_ptr(), stream)
        assert st == 0
        st = lib.logra_sketch_accumulate_noalloc(Xd.data_ptr(), dYd.data_ptr(), n, d, k, r, 5, call,
                                                 S_new.data_ptr(), stream)
        assert st == 0
        torch.cuda.synchronize()
        a, b = S_new.double().cpu().numpy() - 0.5, S_ref.double().cpu().numpy() - 0.5
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL_S


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    import torch
    cap = lib.logra_noalloc_scratch_bytes()
    assert cap > 0
    n, d, k, r = 65536, 1024, 4096, 512           # needs far more scratch than the cap
    assert lib.logra_sketch_workspace_bytes(n, d, k, r, 1) > cap
    X = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")    # never read: rejected first
    S = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    st = lib.logra_sketch_accumulate_noalloc(X.data_ptr(), X.data_ptr(), n, d, k, r, 0, 0, S.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    assert st == 2   # LOGRA_ERR_UNSUPPORTED
