"""LoGRA low-rank gradient sketch + RowAdam apply for GB300 (sm_103a).

The compute lives in liblogra.so (hand-written CUDA kernels behind a C ABI,
``include/logra.h``); this package holds the ctypes binding with the same
entry-point names, the in-tree build script and the seeded input generators.
"""
from .binding import (  # noqa: F401
    LOGRA_BF16, LOGRA_F32, LograError, lib, logra_debug_inject, logra_get_status, logra_launch_count, logra_linear_backward,
    logra_apply_group_workspace_bytes, logra_apply_item, logra_reconstruct, logra_reserve_workspace,
    logra_rowadam_apply, logra_rowadam_apply_bc, logra_rowadam_apply_ex, logra_rowadam_apply_group,
    logra_rowadam_predict, logra_rowadam_predict_bc, logra_set_concurrency, logra_sign_matrix, logra_sketch_accumulate,
    logra_sketch_accumulate_group, logra_sketch_item,
)
