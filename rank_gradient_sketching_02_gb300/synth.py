"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module holds no arithmetic of the method itself: it only draws activations,
gradients, padding masks and weights with the shapes and value distributions of
the workloads, on the host (numpy) or on the device (torch).  Both the CUDA
path and the fp64 oracle consume exactly the bits produced here.

Workloads (attention + MLP projections of decoder layers; the pages compress
only these matrices):

* ``tiny``      one 256 x 512 weight, r=32, 4 microbatches x 128 tokens, fp32;
                X ~ N(0,1), dY ~ N(0, 1e-3^2), 25 of every 128 token rows zeroed.
* ``proj1536``  one 1536 x 1536 weight, r=256, 8 x 4096 tokens, bf16.
* ``layer1p5b`` one 1.5B-class decoder layer (q/o 1536^2, k/v 256x1536,
                gate/up 8960x1536, down 1536x8960), r=256, 16 x 4096 tokens, 3 steps.
* ``model7b``   28 layers of a 7B-class model (q/o 3584^2, k/v 512x3584,
                gate/up 18944x3584, down 3584x18944), r=256, 8 x 8192 tokens.
* ``layers27b`` 4 layers of 27B-class shapes (q/o 5120^2, k/v 1024x5120,
                gate/up 27648x5120, down 5120x27648), r in {128, 256, 512},
                16 x 8192 tokens, 30% padding.

From ``proj1536`` on, dY rows are z * s_t with z ~ N(0,1) and a per-token
lognormal scale s_t = exp(-7 + 1.5 zeta_t), standing in for advantage-weighted
RL gradients; padding rows are zero in both X and dY.

Within a decoder layer the projections that read the same activation share it:
q, k and v read the attention block's input, gate and up the MLP block's input
(``input_group``); o and down read their own.  The benchmark keeps one X per
(layer, input group) and microbatch, and one padding pattern per microbatch.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MATRIX_NAMES = ("q", "k", "v", "o", "gate", "up", "down")

_INPUT_GROUPS = {"q": "attn_in", "k": "attn_in", "v": "attn_in", "o": "attn_out",
                 "gate": "mlp_in", "up": "mlp_in", "down": "mlp_act"}


def input_group(matrix: str) -> str:
    """The activation a projection reads: q/k/v share the attention input, gate/up the MLP input."""
    return _INPUT_GROUPS.get(matrix, matrix)


@dataclass(frozen=True)
class Workload:
    name: str
    matrices: tuple          # ((name, d, k), ...) for one layer
    layers: int
    microbatches: int
    tokens: int              # n per microbatch
    r: int
    dtype: str               # "f32" or "bf16" for X and dY
    mask_frac: float
    dy_kind: str             # "gauss" (N(0, dy_std^2)) or "lognormal"
    dy_std: float = 1.0
    steps: int = 1
    r_sweep: tuple = field(default=())


def _layer(hidden: int, kv: int, ffn: int):
    return (("q", hidden, hidden), ("k", kv, hidden), ("v", kv, hidden),
            ("o", hidden, hidden), ("gate", ffn, hidden), ("up", ffn, hidden),
            ("down", hidden, ffn))


WORKLOADS = {
    "tiny": Workload("tiny", (("w", 256, 512),), 1, 4, 128, 32, "f32",
                     25.0 / 128.0, "gauss", dy_std=1e-3),
    "proj1536": Workload("proj1536", (("w", 1536, 1536),), 1, 8, 4096, 256,
                         "bf16", 0.25, "lognormal"),
    "layer1p5b": Workload("layer1p5b", _layer(1536, 256, 8960), 1, 16, 4096,
                          256, "bf16", 0.25, "lognormal", steps=3),
    "model7b": Workload("model7b", _layer(3584, 512, 18944), 28, 8, 8192, 256,
                        "bf16", 0.25, "lognormal"),
    # one 27B-class / 7B-class gate projection, for kernel profiling at a size well past L2
    "gate27b": Workload("gate27b", (("gate", 27648, 5120),), 1, 2, 8192, 256, "bf16", 0.30, "lognormal"),
    "gate7b": Workload("gate7b", (("gate", 18944, 3584),), 1, 2, 8192, 256, "bf16", 0.25, "lognormal"),
    "layers27b": Workload("layers27b", _layer(5120, 1024, 27648), 4, 16, 8192,
                          256, "bf16", 0.30, "lognormal", r_sweep=(128, 256, 512)),
}

# Hyper-parameters of one RowAdam apply in every workload.
BETA2, EPS, LR_TINY, LR, C = 0.999, 1e-8, 1e-5, 1e-6, 1.0


def matrix_seed(global_seed: int, layer: int, matrix: int) -> int:
    """Per-matrix sign-matrix seed: distinct for every (layer, matrix) pair.

    Without it every same-shaped matrix of a model would share one projection.
    """
    return ((global_seed & 0xFFFFFFFFFFFF) << 16) | ((layer & 0xFFF) << 4) | (matrix & 0xF)


def n_masked(n: int, frac: float) -> int:
    return int(round(n * frac))


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(x) for x in key])))


def host_microbatch(n: int, d: int, k: int, *, dy_kind: str, dy_std: float = 1.0,
                    mask_frac: float = 0.0, key=(0,)):
    """One microbatch on the host as float32 arrays: (X n x k, dY n x d, keep-mask n).

    Padding rows (exactly round(n * mask_frac), chosen by a seeded permutation)
    are zero in X and dY.
    """
    g = _rng(*key)
    X = g.standard_normal((n, k), dtype=np.float32)
    z = g.standard_normal((n, d), dtype=np.float32)
    if dy_kind == "gauss":
        dY = z * np.float32(dy_std)
    elif dy_kind == "lognormal":
        s = np.exp(-7.0 + 1.5 * g.standard_normal(n)).astype(np.float32)
        dY = z * s[:, None]
    else:
        raise ValueError(dy_kind)
    keep = np.ones(n, dtype=bool)
    keep[g.permutation(n)[: n_masked(n, mask_frac)]] = False
    X[~keep] = 0.0
    dY[~keep] = 0.0
    return X, dY, keep


def host_weight(d: int, k: int, std: float = 0.02, key=(0,)) -> np.ndarray:
    return (_rng(*key).standard_normal((d, k), dtype=np.float32) * np.float32(std))


def to_bf16_bits(a: np.ndarray):
    """Round float32 to bfloat16 (round to nearest even) and return it as a torch tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _key_int(x) -> int:
    """Integer key element; names (input groups) enter through their CRC-32."""
    import zlib
    return zlib.crc32(x.encode()) if isinstance(x, str) else int(x)


def _device_generator(key, device):
    import torch
    seed = int(np.random.SeedSequence([_key_int(x) for x in key]).generate_state(1, np.uint64)[0] >> 1)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _device_padding_rows(n: int, mask_frac: float, mb_key, device):
    """The padding rows of one microbatch (shared by every tensor of that microbatch)."""
    import torch
    nm = n_masked(n, mask_frac)
    if not nm:
        return None
    return torch.randperm(n, generator=_device_generator(("pad",) + tuple(mb_key), device), device=device)[:nm]


def device_activations(n: int, k: int, *, mask_frac: float, key, mb_key, dtype=None, device="cuda", out=None):
    """One microbatch's activations X (n x k, N(0,1)) on the device, zero on the microbatch's padding rows."""
    import torch
    X = out if out is not None else torch.empty((n, k), dtype=dtype or torch.bfloat16, device=device)
    X.normal_(0.0, 1.0, generator=_device_generator(key, device))
    drop = _device_padding_rows(n, mask_frac, mb_key, device)
    if drop is not None:
        X.index_fill_(0, drop, 0.0)
    return X


def device_output_grads(n: int, d: int, *, dy_kind: str, dy_std: float = 1.0, mask_frac: float, key, mb_key,
                        dtype=None, device="cuda", out=None):
    """One microbatch's output gradients dY (n x d) on the device, distributed as in ``host_microbatch``,
    zero on the microbatch's padding rows."""
    import torch
    dtype = dtype or torch.bfloat16
    g = _device_generator(key, device)
    dY = out if out is not None else torch.empty((n, d), dtype=dtype, device=device)
    dY.normal_(0.0, 1.0, generator=g)
    if dy_kind == "gauss":
        dY.mul_(dy_std)
    else:
        s = torch.exp(-7.0 + 1.5 * torch.randn(n, generator=g, device=device, dtype=torch.float32))
        dY.mul_(s.to(dtype)[:, None])
    drop = _device_padding_rows(n, mask_frac, mb_key, device)
    if drop is not None:
        dY.index_fill_(0, drop, 0.0)
    return dY


def device_microbatch(n: int, d: int, k: int, *, dy_kind: str, dy_std: float = 1.0,
                      mask_frac: float = 0.0, key=(0,), dtype=None, device="cuda",
                      out_X=None, out_dY=None):
    """One microbatch generated on the device with torch's Philox generator.

    Same distributions as ``host_microbatch``; used where inputs are too large
    to draw on the host.  Writes into ``out_X`` / ``out_dY`` when given.
    """
    import torch
    dtype = dtype or torch.bfloat16
    seed = int(np.random.SeedSequence([int(x) for x in key]).generate_state(1, np.uint64)[0] >> 1)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    X = out_X if out_X is not None else torch.empty((n, k), dtype=dtype, device=device)
    dY = out_dY if out_dY is not None else torch.empty((n, d), dtype=dtype, device=device)
    X.normal_(0.0, 1.0, generator=g)
    dY.normal_(0.0, 1.0, generator=g)
    if dy_kind == "gauss":
        dY.mul_(dy_std)
    else:
        s = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        s = torch.exp(-7.0 + 1.5 * s)
        dY.mul_(s.to(dtype)[:, None])
    nm = n_masked(n, mask_frac)
    if nm:
        drop = torch.randperm(n, generator=g, device=device)[:nm]
        X.index_fill_(0, drop, 0.0)
        dY.index_fill_(0, drop, 0.0)
    return X, dY
