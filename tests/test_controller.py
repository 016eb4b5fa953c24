"""Step-scale controller (host side): the quadratic KL model and the budget."""
import math

import numpy as np
import pytest

from oracle import logra_oracle as O
from rank_gradient_sketching_02_gb300 import controller as K


def test_scale_keeps_predicted_kl_within_budget():
    for kl1 in (1e-6, 0.01, 0.5, 3.0, 1e4):
        for budget in (1e-4, 0.02, 1.0):
            c = K.step_scale(kl1, budget)
            assert 0.0 < c <= 1.0
            assert c * c * kl1 <= budget * (1 + 1e-12)
            if kl1 > budget:
                assert math.isclose(c * c * kl1, budget, rel_tol=1e-12)   # tight when it shrinks
            else:
                assert c == 1.0
    assert K.step_scale(1.0, 0.0) == 0.0


def test_update_norm_is_quadratic_in_c_through_the_oracle():
    # ||dW(c)||^2 = c^2 ||dW(1)||^2, the property the quadratic model rests on
    S = np.random.default_rng(0).standard_normal((6, 32))
    _, _, n1, _ = O.rowadam_apply(np.zeros((6, 128)), S, np.zeros(6), 1, 1, 0.999, 1e-8, 1e-3, 1.0)
    _, _, nc, _ = O.rowadam_apply(np.zeros((6, 128)), S, np.zeros(6), 1, 1, 0.999, 1e-8, 1e-3, 0.3)
    assert math.isclose(nc[1], 0.09 * n1[1], rel_tol=1e-12)


def test_choose_scale_sums_over_matrices():
    norms = [[1.0, 2.0], [5.0, 6.0]]
    kl1 = K.predicted_kl([2.0, 6.0], 0.5)
    assert kl1 == pytest.approx(2.0)
    assert K.choose_scale(norms, 0.5, 0.5) == pytest.approx(0.5)


@pytest.mark.parametrize("kind", ["cosine", "linear"])
def test_annealed_budget_endpoints_and_monotone(kind):
    vals = [K.annealed_budget(s, 100, 0.05, 0.01, kind) for s in range(100)]
    assert vals[0] == pytest.approx(0.05) and vals[-1] == pytest.approx(0.01)
    assert all(a >= b - 1e-15 for a, b in zip(vals, vals[1:]))
    with pytest.raises(ValueError):
        K.annealed_budget(0, 10, 1, 0, "bogus")
