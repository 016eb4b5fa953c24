"""ctypes binding of liblogra.so: the C entry points under the same names.

Argument marshalling only: tensors are checked (device, dtype, contiguity)
and passed as raw device pointers with torch's current CUDA stream; every
step of the computation runs in the library's kernels.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblogra.so")

LOGRA_OK, LOGRA_ERR_INVALID_ARG, LOGRA_ERR_UNSUPPORTED, LOGRA_ERR_CUDA, LOGRA_ERR_TIMEOUT, LOGRA_ERR_NO_DEVICE = range(6)
LOGRA_F32, LOGRA_BF16 = 0, 1

# name -> (restype, argtypes) for every entry point of include/logra.h
_VP, _I, _I64, _U64, _F, _SZ = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_float, C.c_size_t
SIGNATURES = {
    "logra_status_string": (C.c_char_p, [_I]),
    "logra_last_cuda_error": (_I, []),
    "logra_version": (_I, []),
    "logra_launch_count": (_U64, []),
    "logra_sign_matrix": (_I, [_U64, _U64, _I, _I64, _VP, _VP]),
    "logra_sketch_accumulate": (_I, [_VP, _VP, _I, _I64, _I64, _I64, _I, _U64, _U64, _VP, _VP]),
    "logra_rowadam_apply": (_I, [_VP, _VP, _VP, _I64, _I64, _I, _U64, _U64, _F, _F, _F, _F, _VP, _VP]),
    "logra_rowadam_apply_ex": (_I, [_VP, _VP, _VP, _I64, _I64, _I, _U64, _U64, _F, _F, _F, _F, _VP, _VP, _VP,
                                    _VP]),
    "logra_rowadam_apply_bc": (_I, [_VP, _VP, _VP, _I64, _I64, _I, _U64, _U64, _F, _F, _F, _F, _I64, _VP, _VP,
                                    _VP, _VP]),
    "logra_rowadam_predict": (_I, [_VP, _VP, _I64, _I64, _I, _U64, _U64, _F, _F, _F, _VP, _VP]),
    "logra_rowadam_predict_bc": (_I, [_VP, _VP, _I64, _I64, _I, _U64, _U64, _F, _F, _F, _I64, _VP, _VP]),
    "logra_reconstruct": (_I, [_VP, _I64, _I64, _I, _U64, _U64, _VP, _I, _I, _VP]),
    "logra_get_status": (_I, [_VP]),
    "logra_reserve_workspace": (_I, [_SZ, _VP]),
    "logra_sketch_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "logra_apply_workspace_bytes": (_SZ, [_I64, _I64, _I]),
    "logra_debug_inject": (_I, [_I, _U64]),
    "logra_set_concurrency": (_I, [_I]),
    "logra_sketch_accumulate_noalloc": (_I, [_VP, _VP, _I64, _I64, _I64, _I, _U64, _U64, _VP, _VP]),
    "logra_noalloc_scratch_bytes": (_SZ, []),
    "logra_linear_backward": (_I, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I, _U64, _U64, _VP, _VP]),
}



class logra_apply_item(C.Structure):
    """One matrix of logra_rowadam_apply_group (the C struct of the same name)."""
    _fields_ = [("W", _VP), ("S", _VP), ("v", _VP), ("d", _I64), ("k", _I64), ("seed", _U64),
                ("lr", _F), ("c", _F), ("norms_out", _VP), ("W_bf16_out", _VP), ("sync_sketch_out", _VP),
                ("t", _I64)]


class logra_sketch_item(C.Structure):
    """One sketch of logra_sketch_accumulate_group (the C struct of the same name)."""
    _fields_ = [("X", _VP), ("dY", _VP), ("S", _VP), ("d", _I64), ("k", _I64), ("seed", _U64)]


SIGNATURES["logra_rowadam_apply_group"] = (_I, [C.POINTER(logra_apply_item), _I, _I, _U64, _F, _F, _VP])
SIGNATURES["logra_sketch_accumulate_group"] = (_I, [C.POINTER(logra_sketch_item), _I, _I64, _I, _U64, _VP])
SIGNATURES["logra_apply_group_workspace_bytes"] = (_SZ, [C.POINTER(logra_apply_item), _I, _I])

_lib = None
_lock = threading.Lock()


class LograError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().logra_status_string(status).decode()
        if status == LOGRA_ERR_CUDA:
            msg += f" (cudaError {lib().logra_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {status}]")


def lib():
    """Load liblogra.so (built in-tree by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"liblogra.so not built ({LIB_PATH}); run the package's build.py")
                h = C.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    f = getattr(h, name)
                    f.restype, f.argtypes = res, args
                _lib = h
    return _lib


def _check(st: int, where: str):
    if st != LOGRA_OK:
        raise LograError(st, where)


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, name, dtypes=None, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _in_dtype(t):
    import torch
    return {torch.float32: LOGRA_F32, torch.bfloat16: LOGRA_BF16}[t.dtype]


def logra_sign_matrix(seed: int, step: int, r: int, k: int, A_out=None, stream=None):
    import torch
    if A_out is None:
        A_out = torch.empty((r, k), dtype=torch.float32, device="cuda")
    p = _dev(A_out, "A_out", (torch.float32,), (r, k))
    _check(lib().logra_sign_matrix(seed, step, r, k, p, _stream(stream)), "logra_sign_matrix")
    return A_out


def logra_sketch_accumulate(X, dY, S, seed: int, step: int, stream=None):
    """S (d x r fp32) += dY^T (X A^T) for one microbatch; X n x k, dY n x d."""
    import torch
    n, k = X.shape
    d, r = S.shape
    dt = (torch.float32, torch.bfloat16)
    px = _dev(X, "X", dt)
    py = _dev(dY, "dY", (X.dtype,), (n, d))
    ps = _dev(S, "S", (torch.float32,))
    _check(lib().logra_sketch_accumulate(px, py, _in_dtype(X), n, d, k, r, seed, step, ps, _stream(stream)),
           "logra_sketch_accumulate")
    return S


def logra_linear_backward(dY, W=None, dX=None, X=None, S=None, seed: int = 0, step: int = 0, stream=None):
    """Linear-layer backward for one microbatch: dX = dY W (bf16) and S += dY^T (X A^T).

    dY: n x d bf16; W: d x k bf16 and dX: n x k bf16 (out), or both None for the sketch only;
    X: n x k bf16 and S: d x r fp32, or both None for dX only."""
    import torch
    bf = (torch.bfloat16,)
    n, d = dY.shape
    if dX is not None:
        k = dX.shape[1]
    elif X is not None:
        k = X.shape[1]
    else:
        raise ValueError("dX and S are both None: nothing to compute")
    r = 32
    py = _dev(dY, "dY", bf)
    pw = _dev(W, "W", bf, (d, k)) if dX is not None else None
    pdx = _dev(dX, "dX", bf, (n, k)) if dX is not None else None
    px = _dev(X, "X", bf, (n, k)) if S is not None else None
    if S is not None:
        r = S.shape[1]
        ps = _dev(S, "S", (torch.float32,), (d, r))
    else:
        ps = None
    _check(lib().logra_linear_backward(px, py, pw, pdx, n, d, k, r, seed, step, ps, _stream(stream)),
           "logra_linear_backward")
    return dX


def logra_sketch_accumulate_group(items, step: int, stream=None):
    """logra_sketch_accumulate for several bf16 sketches of one n and r from one caller stream.

    items: sequence of dicts with X (n x k), dY (n x d) bf16 CUDA tensors, S (d x r fp32) and seed;
    the library spreads them over its own side streams and joins them back into the stream."""
    import torch
    items = list(items)
    arr = (logra_sketch_item * max(1, len(items)))()
    n = r = None
    for i, m in enumerate(items):
        X, dY, S = m["X"], m["dY"], m["S"]
        if n is None:
            n, r = X.shape[0], S.shape[1]
        elif X.shape[0] != n or S.shape[1] != r:
            raise ValueError("every sketch of a group has the same token count n and rank r")
        k, d = X.shape[1], S.shape[0]
        bf = (torch.bfloat16,)
        arr[i] = logra_sketch_item(_dev(X, "X", bf), _dev(dY, "dY", bf, (n, d)), _dev(S, "S", (torch.float32,)),
                                   d, k, int(m["seed"]))
    _check(lib().logra_sketch_accumulate_group(arr, len(items), n or 0, r or 32, step, _stream(stream)),
           "logra_sketch_accumulate_group")


def logra_rowadam_apply(W, S, v, seed: int, step: int, beta2: float, eps: float, lr: float, c: float,
                        norms_out=None, stream=None):
    import torch
    d, k = W.shape
    r = S.shape[1]
    f32 = (torch.float32,)
    pw = _dev(W, "W", f32)
    ps = _dev(S, "S", f32, (d, r))
    pv = _dev(v, "v", f32, (d,))
    pn = _dev(norms_out, "norms_out", (torch.float64,), (2,)) if norms_out is not None else None
    _check(lib().logra_rowadam_apply(pw, ps, pv, d, k, r, seed, step, beta2, eps, lr, c, pn, _stream(stream)),
           "logra_rowadam_apply")
    return W


def logra_rowadam_apply_ex(W, S, v, seed: int, step: int, beta2: float, eps: float, lr: float, c: float,
                           norms_out=None, W_bf16_out=None, sync_sketch_out=None, stream=None):
    import torch
    d, k = W.shape
    r = S.shape[1]
    f32 = (torch.float32,)
    pw = _dev(W, "W", f32)
    ps = _dev(S, "S", f32, (d, r))
    pv = _dev(v, "v", f32, (d,))
    pn = _dev(norms_out, "norms_out", (torch.float64,), (2,)) if norms_out is not None else None
    pb = _dev(W_bf16_out, "W_bf16_out", (torch.bfloat16,), (d, k)) if W_bf16_out is not None else None
    pq = _dev(sync_sketch_out, "sync_sketch_out", f32, (d, r)) if sync_sketch_out is not None else None
    _check(lib().logra_rowadam_apply_ex(pw, ps, pv, d, k, r, seed, step, beta2, eps, lr, c, pn, pb, pq,
                                        _stream(stream)), "logra_rowadam_apply_ex")
    return W


def _apply_items(items):
    """items: sequence of dicts with W, S, v, seed, lr, c and optional norms_out, W_bf16_out,
    sync_sketch_out (CUDA tensors as for logra_rowadam_apply_ex).  Returns (ctypes array, r)."""
    import torch
    f32 = (torch.float32,)
    arr = (logra_apply_item * max(1, len(items)))()
    r = None
    for i, m in enumerate(items):
        W, S, v = m["W"], m["S"], m["v"]
        d, k = W.shape
        if r is None:
            r = S.shape[1]
        elif S.shape[1] != r:
            raise ValueError("every matrix of a group has the same rank r")
        nm, wb, sq = m.get("norms_out"), m.get("W_bf16_out"), m.get("sync_sketch_out")
        arr[i] = logra_apply_item(
            _dev(W, "W", f32), _dev(S, "S", f32, (d, r)), _dev(v, "v", f32, (d,)), d, k, int(m["seed"]),
            float(m["lr"]), float(m["c"]),
            _dev(nm, "norms_out", (torch.float64,), (2,)) if nm is not None else None,
            _dev(wb, "W_bf16_out", (torch.bfloat16,), (d, k)) if wb is not None else None,
            _dev(sq, "sync_sketch_out", f32, (d, r)) if sq is not None else None, int(m.get("t", 0)))
    return arr, (r if r is not None else 32)


def logra_rowadam_apply_group(items, step: int, beta2: float, eps: float, stream=None):
    """logra_rowadam_apply_ex over several matrices of one rank in grouped launches."""
    arr, r = _apply_items(items)
    _check(lib().logra_rowadam_apply_group(arr, len(items), r, step, beta2, eps, _stream(stream)),
           "logra_rowadam_apply_group")


def logra_apply_group_workspace_bytes(items) -> int:
    arr, r = _apply_items(items)
    return int(lib().logra_apply_group_workspace_bytes(arr, len(items), r))


def logra_rowadam_apply_bc(W, S, v, seed: int, step: int, beta2: float, eps: float, lr: float, c: float, t: int,
                           norms_out=None, W_bf16_out=None, sync_sketch_out=None, stream=None):
    """logra_rowadam_apply_ex with Adam's bias correction for the t-th update (t >= 1)."""
    import torch
    d, k = W.shape
    r = S.shape[1]
    f32 = (torch.float32,)
    pw = _dev(W, "W", f32)
    ps = _dev(S, "S", f32, (d, r))
    pv = _dev(v, "v", f32, (d,))
    pn = _dev(norms_out, "norms_out", (torch.float64,), (2,)) if norms_out is not None else None
    pb = _dev(W_bf16_out, "W_bf16_out", (torch.bfloat16,), (d, k)) if W_bf16_out is not None else None
    pq = _dev(sync_sketch_out, "sync_sketch_out", f32, (d, r)) if sync_sketch_out is not None else None
    _check(lib().logra_rowadam_apply_bc(pw, ps, pv, d, k, r, seed, step, beta2, eps, lr, c, t, pn, pb, pq,
                                        _stream(stream)), "logra_rowadam_apply_bc")
    return W


def logra_rowadam_predict_bc(S, v, k: int, seed: int, step: int, beta2: float, eps: float, lr: float, t: int,
                             norms_out, stream=None):
    import torch
    d, r = S.shape
    f32 = (torch.float32,)
    ps = _dev(S, "S", f32)
    pv = _dev(v, "v", f32, (d,))
    pn = _dev(norms_out, "norms_out", (torch.float64,), (2,))
    _check(lib().logra_rowadam_predict_bc(ps, pv, d, k, r, seed, step, beta2, eps, lr, t, pn, _stream(stream)),
           "logra_rowadam_predict_bc")
    return norms_out


def logra_rowadam_predict(S, v, k: int, seed: int, step: int, beta2: float, eps: float, lr: float,
                          norms_out, stream=None):
    import torch
    d, r = S.shape
    f32 = (torch.float32,)
    ps = _dev(S, "S", f32)
    pv = _dev(v, "v", f32, (d,))
    pn = _dev(norms_out, "norms_out", (torch.float64,), (2,))
    _check(lib().logra_rowadam_predict(ps, pv, d, k, r, seed, step, beta2, eps, lr, pn, _stream(stream)),
           "logra_rowadam_predict")
    return norms_out


def logra_reconstruct(S, k: int, seed: int, step: int, out, accumulate: bool = False, stream=None):
    import torch
    d, r = S.shape
    ps = _dev(S, "S", (torch.float32,))
    po = _dev(out, "out", (torch.float32, torch.bfloat16), (d, k))
    _check(lib().logra_reconstruct(ps, d, k, r, seed, step, po, _in_dtype(out), int(bool(accumulate)),
                                   _stream(stream)), "logra_reconstruct")
    return out


def logra_get_status(stream=None) -> int:
    return lib().logra_get_status(_stream(stream))


def logra_reserve_workspace(nbytes: int, stream=None):
    _check(lib().logra_reserve_workspace(nbytes, _stream(stream)), "logra_reserve_workspace")


def logra_launch_count() -> int:
    return int(lib().logra_launch_count())


def logra_set_concurrency(streams: int):
    _check(lib().logra_set_concurrency(int(streams)), "logra_set_concurrency")


def logra_debug_inject(fault: int, timeout_cycles: int = 0):
    _check(lib().logra_debug_inject(fault, timeout_cycles), "logra_debug_inject")
