"""The C ABI library builds, loads without a GPU and exports what the header declares."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "logra.h")


@pytest.fixture(scope="module")
def lib():
    from rank_gradient_sketching_02_gb300 import build as B
    B.build()
    from rank_gradient_sketching_02_gb300 import binding
    return binding.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(logra_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for must in ("logra_sketch_accumulate", "logra_rowadam_apply", "logra_reconstruct", "logra_sign_matrix"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    import ctypes
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_binding_covers_every_declared_symbol():
    from rank_gradient_sketching_02_gb300 import binding
    assert sorted(binding.SIGNATURES) == header_functions()


def test_host_only_calls(lib):
    assert lib.logra_version() >> 16 == 1
    for st in range(6):
        assert lib.logra_status_string(st)
    assert lib.logra_status_string(99) == b"unknown status"
    assert lib.logra_sketch_workspace_bytes(8192, 1536, 1536, 256, 1) >= 8192 * 256 * 4
    # fp32: the bf16 scratch of the 4n stacked tokens, then the stacked bf16 planes of X and dY
    assert (lib.logra_sketch_workspace_bytes(8192, 1536, 1536, 256, 0)
            >= lib.logra_sketch_workspace_bytes(4 * 8192, 1536, 1536, 256, 1) + 8 * 8192 * (1536 + 1536))
    assert lib.logra_sketch_workspace_bytes((1 << 28) + 1, 8, 8, 32, 1) == 0
    assert lib.logra_sketch_workspace_bytes(0, 8, 8, 32, 1) == 0
    assert lib.logra_apply_workspace_bytes(1536, 1536, 256) > 0


def test_bad_arguments_rejected_before_any_cuda_call(lib):
    from rank_gradient_sketching_02_gb300.binding import LOGRA_ERR_INVALID_ARG, LOGRA_ERR_UNSUPPORTED
    # null / negative / bad dtype / bad rank / unaligned: no device work is attempted
    assert lib.logra_sketch_accumulate(None, None, 1, 16, 8, 8, 32, 0, 0, None, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate(16, 16, 7, 16, 8, 8, 32, 0, 0, 16, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate(16, 16, 1, 16, 12, 8, 32, 0, 0, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_sketch_accumulate(16, 16, 1, 16, 8, 8, 48, 0, 0, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_sketch_accumulate(16, 18, 1, 16, 8, 8, 32, 0, 0, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_sketch_accumulate(16, 16, 1, 0, 8, 8, 32, 0, 0, 16, None) == 0   # n == 0: no-op
    assert lib.logra_sign_matrix(0, 0, 544, 8, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_reconstruct(16, 8, 8, 32, 0, 0, 16, 5, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_rowadam_predict(16, 16, 8, 8, 32, 0, 0, 0.9, 1e-8, 1e-3, None, None) == LOGRA_ERR_INVALID_ARG
    # linear backward: neither output, a misaligned dX, a bad rank with S, n too large, n == 0 (no-op)
    assert lib.logra_linear_backward(16, 16, 16, None, 64, 64, 64, 32, 0, 0, None, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_linear_backward(None, 16, 16, 18, 64, 64, 64, 32, 0, 0, None, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_linear_backward(16, 16, None, None, 64, 64, 64, 48, 0, 0, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_linear_backward(16, 16, 16, 16, 2**31, 64, 64, 32, 0, 0, 16, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_linear_backward(16, 16, None, 16, 64, 64, 64, 32, 0, 0, None, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_linear_backward(16, 16, 16, 16, 0, 64, 64, 32, 0, 0, 16, None) == 0


def _items(binding, shapes, W=16, S=16, v=16):
    arr = (binding.logra_apply_item * max(1, len(shapes)))()
    for i, (d, k) in enumerate(shapes):
        arr[i] = binding.logra_apply_item(W, S, v, d, k, i, 1e-3, 1.0, None, None, None)
    return arr


def test_group_workspace_is_the_largest_launch_group(lib):
    from rank_gradient_sketching_02_gb300 import binding
    def single(d, k):
        return (lib.logra_apply_workspace_bytes(d, k, 256) + 255) // 256 * 256
    small = [(512, 3584)] * 3 + [(3584, 3584)] * 5                     # one launch group of 8
    assert lib.logra_apply_group_workspace_bytes(_items(binding, small), 8, 256) == sum(single(*s) for s in small)
    big = small + [(18944, 3584)] * 2                                   # groups of 8 and 2
    want = max(sum(single(*s) for s in big[:8]), sum(single(*s) for s in big[8:]))
    assert lib.logra_apply_group_workspace_bytes(_items(binding, big), 10, 256) == want
    assert lib.logra_apply_group_workspace_bytes(_items(binding, small), 8, 48) == 0   # bad rank
    assert lib.logra_apply_group_workspace_bytes(None, 8, 256) == 0


def test_group_bad_arguments_rejected_before_any_cuda_call(lib):
    from rank_gradient_sketching_02_gb300.binding import LOGRA_ERR_INVALID_ARG, LOGRA_ERR_UNSUPPORTED
    from rank_gradient_sketching_02_gb300 import binding
    ok = [(64, 64), (128, 64)]
    assert lib.logra_rowadam_apply_group(_items(binding, ok), 0, 256, 0, 0.9, 1e-8, None) == 0   # no-op
    assert lib.logra_rowadam_apply_group(None, 2, 256, 0, 0.9, 1e-8, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_rowadam_apply_group(_items(binding, ok), -1, 256, 0, 0.9, 1e-8, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_rowadam_apply_group(_items(binding, ok), 2, 48, 0, 0.9, 1e-8, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_rowadam_apply_group(_items(binding, ok, W=None), 2, 256, 0, 0.9, 1e-8, None) == \
        LOGRA_ERR_INVALID_ARG
    assert lib.logra_rowadam_apply_group(_items(binding, [(64, 64), (12, 64)]), 2, 256, 0, 0.9, 1e-8, None) == \
        LOGRA_ERR_UNSUPPORTED
    assert lib.logra_rowadam_apply_group(_items(binding, ok, S=24), 2, 256, 0, 0.9, 1e-8, None) == \
        LOGRA_ERR_UNSUPPORTED


def test_bias_correction_arguments_rejected_before_any_cuda_call(lib):
    from rank_gradient_sketching_02_gb300.binding import LOGRA_ERR_INVALID_ARG
    from rank_gradient_sketching_02_gb300 import binding
    args = (16, 16, 16, 64, 64, 32, 0, 0)
    assert lib.logra_rowadam_apply_bc(*args, 0.999, 1e-8, 1e-3, 1.0, -1, None, None, None, None) == \
        LOGRA_ERR_INVALID_ARG                                            # t < 0
    assert lib.logra_rowadam_apply_bc(*args, 1.0, 1e-8, 1e-3, 1.0, 2, None, None, None, None) == \
        LOGRA_ERR_INVALID_ARG                                            # beta2 = 1: 1 - beta2^t = 0
    assert lib.logra_rowadam_predict_bc(16, 16, 64, 64, 32, 0, 0, 1.5, 1e-8, 1e-3, 1, 16, None) == \
        LOGRA_ERR_INVALID_ARG
    arr = _items(binding, [(64, 64)])
    arr[0].t = -3
    assert lib.logra_rowadam_apply_group(arr, 1, 256, 0, 0.9, 1e-8, None) == LOGRA_ERR_INVALID_ARG


def test_concurrency_hint_is_validated(lib):
    from rank_gradient_sketching_02_gb300.binding import LOGRA_ERR_INVALID_ARG
    assert lib.logra_set_concurrency(0) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_set_concurrency(65) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_set_concurrency(4) == 0
    assert lib.logra_set_concurrency(1) == 0


def test_sketch_group_bad_arguments_rejected_before_any_cuda_call(lib):
    from rank_gradient_sketching_02_gb300.binding import LOGRA_ERR_INVALID_ARG, LOGRA_ERR_UNSUPPORTED
    from rank_gradient_sketching_02_gb300 import binding

    def items(shapes, X=4096, dY=8192, S=16384):
        arr = (binding.logra_sketch_item * len(shapes))()
        for i, (d, k) in enumerate(shapes):
            arr[i] = binding.logra_sketch_item(X, dY, S, d, k, 7)
        return arr

    ok = [(64, 64), (128, 72)]
    assert lib.logra_sketch_accumulate_group(items(ok), 0, 128, 256, 0, None) == 0           # no-op
    assert lib.logra_sketch_accumulate_group(items(ok), 2, 0, 256, 0, None) == 0             # n == 0
    assert lib.logra_sketch_accumulate_group(None, 2, 128, 256, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate_group(items(ok), -1, 128, 256, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate_group(items(ok), 2, -5, 256, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate_group(items(ok), 2, 128, 40, 0, None) == LOGRA_ERR_UNSUPPORTED
    assert lib.logra_sketch_accumulate_group(items([(64, 64), (12, 64)]), 2, 128, 256, 0, None) == \
        LOGRA_ERR_UNSUPPORTED
    assert lib.logra_sketch_accumulate_group(items(ok, S=0), 2, 128, 256, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate_group(items(ok, X=0), 2, 128, 256, 0, None) == LOGRA_ERR_INVALID_ARG
    assert lib.logra_sketch_accumulate_group(items(ok, dY=8200), 2, 128, 256, 0, None) == LOGRA_ERR_UNSUPPORTED
