"""Plain fp64 CPU oracle for the LoGRA sketch / RowAdam hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library (no kernels, headers, constant tables or helpers); the only
thing both sides receive in common is the seeded synthetic input.

Every function follows the plain definition of the quantity it computes, in
fp64, with one numpy library primitive (a matmul, a sum) per step and no
blocking, fusion or reordering beyond that definition.

Notation (LoGRA: Scaling LLM Reinforcement Learning with Low-Rank Gradient
Sketches, academy.dair.ai summary, "Gradient sketches"; theclarity.today
write-up, "Why it matters"):

* W      d x k projection weight (rows = output channels, nn.Linear layout)
* X      n x k microbatch activations (one row per token)
* dY     n x d microbatch output gradients
* G      = dY^T X, the d x k weight gradient (never formed on the hot path)
* Sigma  r x k random-sign matrix, entries +-1, redrawn each step and held
         fixed across the step's microbatches
* A      = Sigma / sqrt(r)
* S      d x r sketch, S = G A^T, accumulated over microbatches
* Ghat   = S A, the d x k reconstruction used at apply time
* v      d per-row second moment of RowAdam (no first moment)

Readings taken where the pages are silent (each is listed with its reason in
the design notes of this repository):

* the sign generator: SplitMix64 (Steele, Lea & Flood, "Fast Splittable
  Pseudorandom Number Generators", OOPSLA 2014).  The step key is output
  number step+1 of SplitMix64 seeded with ``seed``; word (i, w) of row i of
  Sigma is the SplitMix64 finaliser of ``key XOR (i << 32 | w)``; entry
  Sigma[i, j] is -1 when bit (j mod 64) of word (i, j div 64) is set, else +1.
* the sign scale is 1/sqrt(r), so diag(A^T A) == 1 and E[A^T A] = I.
* "row magnitude" is the mean over the k columns of Ghat_ij^2.
* v is updated with the current Ghat before it scales the step; no bias
  correction by default (an optional variant divides v by 1 - beta2^t for the
  step only), no weight decay; eps sits inside the square root.
* microbatch contributions are summed; padding tokens are zero rows of X and
  dY supplied by the caller.
* ||dW||^2 is taken over the intended update -lr*c*Ghat/sqrt(v+eps), not over
  a difference of rounded weights.

parity pinned: every function here is checked by ``tests/test_oracle_pins.py``
against published generator outputs, brute-force sums, closed forms,
linearity and a Monte-Carlo unbiasedness bound.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "MASK64", "GAMMA", "splitmix64_finalize", "splitmix64_outputs",
    "step_key", "sign_words", "sign_matrix", "projection_matrix",
    "projection_matrix_fp32", "sketch_accumulate", "sketch_columns",
    "reconstruct", "rowadam_apply", "rowadam_rows", "gram_matrix",
    "sync_sketch", "bias_corrected", "input_gradient", "linear_backward",
]

MASK64 = (1 << 64) - 1
# SplitMix64 increment (the 64-bit golden-ratio constant of the published generator).
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64_finalize(z):
    """SplitMix64 output function (Steele, Lea & Flood 2014), on uint64 arrays.

    z ^= z >> 30; z *= M1; z ^= z >> 27; z *= M2; z ^= z >> 31  (mod 2^64).
    """
    z = np.array(z, dtype=np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def splitmix64_outputs(seed: int, count: int) -> np.ndarray:
    """First ``count`` outputs of SplitMix64 seeded with ``seed``.

    The generator's state after n calls is seed + n*GAMMA; output n is the
    finaliser of that state.
    """
    n = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        states = np.uint64(seed & MASK64) + n * GAMMA
    return splitmix64_finalize(states)


def step_key(seed: int, step: int) -> np.uint64:
    """Key of the sign matrix for (seed, step): SplitMix64 output number step+1.

    A new key per step gives the "redrawn each step" projection (academy.dair.ai
    summary, "Gradient sketches"); every microbatch of the step reuses it.
    """
    with np.errstate(over="ignore"):
        state = np.uint64(seed & MASK64) + np.uint64((step + 1) & MASK64) * GAMMA
    return splitmix64_finalize(state)[()]


def sign_words(seed: int, step: int, r: int, k: int) -> np.ndarray:
    """r x ceil(k/64) uint64 words; bit b of word (i, w) is the sign bit of Sigma[i, 64w+b]."""
    nw = (k + 63) // 64
    i = np.arange(r, dtype=np.uint64)[:, None]
    w = np.arange(nw, dtype=np.uint64)[None, :]
    counter = (i << np.uint64(32)) | w
    return splitmix64_finalize(step_key(seed, step) ^ counter)


def sign_matrix(seed: int, step: int, r: int, k: int) -> np.ndarray:
    """Sigma (r x k, int8 entries +-1): -1 where the sign bit is set."""
    words = sign_words(seed, step, r, k)
    j = np.arange(k)
    bits = (words[:, j // 64] >> (j % 64).astype(np.uint64)) & np.uint64(1)
    return (1 - 2 * bits.astype(np.int64)).astype(np.int8)


def projection_matrix(seed: int, step: int, r: int, k: int) -> np.ndarray:
    """A = Sigma / sqrt(r) in fp64 (r x k)."""
    return sign_matrix(seed, step, r, k).astype(np.float64) / np.sqrt(r)


def projection_matrix_fp32(seed: int, step: int, r: int, k: int) -> np.ndarray:
    """A as fp32: Sigma * fl32(1/sqrt(r)), the exact bits a float32 sign matrix holds."""
    scale = np.float32(1.0 / np.sqrt(np.float64(r)))
    return sign_matrix(seed, step, r, k).astype(np.float32) * scale


def sketch_accumulate(S: np.ndarray, X: np.ndarray, dY: np.ndarray,
                      seed: int, step: int, r: int) -> np.ndarray:
    """One microbatch of the sketch: returns S + dY^T (X A^T).

    This is G A^T with G = dY^T X (theclarity.today write-up, "Why it
    matters": the sketch S = G * A^T), computed without forming G.
    """
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    A = projection_matrix(seed, step, r, X.shape[1])
    P = X @ A.T                     # n x r
    return np.asarray(S, dtype=np.float64) + dY.T @ P


def input_gradient(dY: np.ndarray, W: np.ndarray) -> np.ndarray:
    """dX = dY W (n x k): the gradient with respect to the input of a Linear
    layer Y = X W^T.  The method leaves this half of the backward pass as it
    is; only the weight gradient dY^T X is replaced by the sketch
    (theclarity.today write-up, "Why it matters")."""
    return np.asarray(dY, dtype=np.float64) @ np.asarray(W, dtype=np.float64)


def linear_backward(S: np.ndarray, X: np.ndarray, dY: np.ndarray, W: np.ndarray,
                    seed: int, step: int, r: int):
    """One microbatch of a Linear layer's backward as the method runs it:
    returns (dX, S + dY^T (X A^T)), the input gradient and the updated sketch,
    with no d x k gradient buffer (academy.dair.ai summary, "Gradient
    sketches")."""
    return input_gradient(dY, W), sketch_accumulate(S, X, dY, seed, step, r)


def sketch_columns(X: np.ndarray, dY: np.ndarray, seed: int, step: int,
                   r: int, cols) -> np.ndarray:
    """Columns ``cols`` of one microbatch's sketch dY^T (X A^T), as d x len(cols).

    Column c of the sketch only needs row c of A, so full-size cases can be
    checked column by column.
    """
    X = np.asarray(X, dtype=np.float64)
    A = projection_matrix(seed, step, r, X.shape[1])[np.asarray(cols)]
    P = X @ A.T                     # n x len(cols)
    return np.asarray(dY, dtype=np.float64).T @ P


def reconstruct(S: np.ndarray, seed: int, step: int, k: int) -> np.ndarray:
    """Ghat = S A (d x k): the full-size update direction rebuilt from the sketch."""
    S = np.asarray(S, dtype=np.float64)
    return S @ projection_matrix(seed, step, S.shape[1], k)


def bias_corrected(v_new: np.ndarray, beta2: float, t: int) -> np.ndarray:
    """Adam's bias correction of the second moment, v / (1 - beta2^t), for the
    t-th update (t >= 1); t = 0 means no correction (the default RowAdam).

    Adam divides its running averages by 1 - beta^t because they start at zero
    (Kingma & Ba, "Adam: A Method for Stochastic Optimization", ICLR 2015,
    Algorithm 1); the pages name Adam's correction (academy.dair.ai summary)
    but leave RowAdam's open, so the corrected form is an optional variant.
    """
    v_new = np.asarray(v_new, dtype=np.float64)
    if t == 0:
        return v_new
    return v_new / (1.0 - beta2 ** t)


def rowadam_apply(W: np.ndarray, S: np.ndarray, v: np.ndarray, seed: int,
                  step: int, beta2: float, eps: float, lr: float, c: float, t: int = 0):
    """RowAdam step from the sketch.

    Ghat = S A; m_i = mean_j Ghat_ij^2; v_i <- beta2 v_i + (1-beta2) m_i;
    dW_ij = -lr c Ghat_ij / sqrt(v_i + eps); W <- W + dW.
    RowAdam keeps one squared-row-magnitude statistic per row and no first
    moment (theclarity.today write-up, "What happened" and "Why it matters").
    With t >= 1 the step uses the bias-corrected v / (1 - beta2^t) in place of
    v (the stored v stays uncorrected).

    Returns (W_new, v_new, norms, dW) with norms = (||S||_F^2, ||dW||_F^2).
    """
    S = np.asarray(S, dtype=np.float64)
    k = np.asarray(W).shape[1]
    Ghat = reconstruct(S, seed, step, k)
    m = np.mean(Ghat * Ghat, axis=1)
    v_new = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * m
    dW = -lr * c * Ghat / np.sqrt(bias_corrected(v_new, beta2, t) + eps)[:, None]
    W_new = np.asarray(W, dtype=np.float64) + dW
    norms = np.array([np.sum(S * S), np.sum(dW * dW)])
    return W_new, v_new, norms, dW


def rowadam_rows(S_rows: np.ndarray, v_rows: np.ndarray, k: int, seed: int,
                 step: int, beta2: float, eps: float, lr: float, c: float, t: int = 0):
    """RowAdam on a subset of rows (rows are independent given S): (v_new, dW, Ghat)."""
    S_rows = np.asarray(S_rows, dtype=np.float64)
    Ghat = reconstruct(S_rows, seed, step, k)
    m = np.mean(Ghat * Ghat, axis=1)
    v_new = beta2 * np.asarray(v_rows, dtype=np.float64) + (1.0 - beta2) * m
    dW = -lr * c * Ghat / np.sqrt(bias_corrected(v_new, beta2, t) + eps)[:, None]
    return v_new, dW, Ghat


def sync_sketch(S: np.ndarray, v_new: np.ndarray, eps: float, lr: float,
                c: float, beta2: float = 0.0, t: int = 0) -> np.ndarray:
    """Row-scaled sketch S'_i = -lr c S_i / sqrt(v_i + eps).

    The row scaling commutes with the right product by A, so S' A is the
    applied update: a rollout worker rebuilds dW from the d x r payload
    (academy.dair.ai summary: the update is the product of two small matrices,
    which makes policy synchronisation cheaper).
    """
    S = np.asarray(S, dtype=np.float64)
    return -lr * c * S / np.sqrt(bias_corrected(v_new, beta2, t) + eps)[:, None]


def gram_matrix(seed: int, step: int, r: int, k: int) -> np.ndarray:
    """M = Sigma Sigma^T (r x r, exact integers), so that ||(S A)_i||^2 = S_i M S_i^T / r."""
    Sg = sign_matrix(seed, step, r, k).astype(np.int64)
    return Sg @ Sg.T
