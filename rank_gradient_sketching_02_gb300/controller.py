"""Caller-side step scale from the library's norms (predicted-KL step control).

The pages say that before each update LoGRA predicts the resulting change of
the policy's KL divergence from the sketch itself and scales the step so it
stays within a budget that is annealed over training (academy.dair.ai summary,
"Step control"; theclarity.today write-up, "What happened" and "Why it
matters"), and that the shrink factor is closed-form (eyestech.in, "Predicted-
KL Step Control").  The page that starts to give the formula is cut off before
it, so this module takes the plainest reading that the rest supports:

* a local quadratic model, KL(c) = c^2 KL(1), where c scales the whole update
  (dW is linear in c, so ||dW(c)||^2 = c^2 ||dW(1)||^2 exactly);
* KL(1) = 0.5 * fisher_scale * sum over matrices of ||dW(1)||^2, i.e. an
  isotropic Fisher whose scale the caller calibrates (the empirical Fisher
  itself is not on the pages);
* c = min(1, sqrt(budget / KL(1))), so the predicted KL never exceeds the
  budget and an update already inside it is left alone;
* budget_t annealed from `start` to `end` over `total` steps (cosine or
  linear; the pages name no schedule).

These are host-side scalars computed from the norms that
logra_rowadam_predict returns; no kernel is involved.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence


def predicted_kl(update_sq_norms: Iterable[float], fisher_scale: float) -> float:
    """KL(1) = 0.5 * fisher_scale * sum ||dW(1)||^2 over the compressed matrices."""
    return 0.5 * float(fisher_scale) * float(sum(update_sq_norms))


def step_scale(kl_at_unit_step: float, budget: float) -> float:
    """Largest c in (0, 1] with c^2 * KL(1) <= budget."""
    if budget <= 0.0:
        return 0.0
    if kl_at_unit_step <= budget:
        return 1.0
    return math.sqrt(budget / kl_at_unit_step)


def annealed_budget(step: int, total: int, start: float, end: float, kind: str = "cosine") -> float:
    """KL budget at `step` of `total`, moving from `start` to `end`."""
    if total <= 1:
        return float(end)
    t = min(max(step / (total - 1), 0.0), 1.0)
    if kind == "linear":
        w = t
    elif kind == "cosine":
        w = 0.5 * (1.0 - math.cos(math.pi * t))
    else:
        raise ValueError(kind)
    return float(start + (end - start) * w)


def choose_scale(norms_per_matrix: Sequence[Sequence[float]], fisher_scale: float, budget: float) -> float:
    """c for one optimiser step from the [||S||^2, ||dW(1)||^2] pairs of every matrix."""
    return step_scale(predicted_kl((n[1] for n in norms_per_matrix), fisher_scale), budget)
