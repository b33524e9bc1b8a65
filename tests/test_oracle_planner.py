"""Pins for the oracle's alpha / gamma planner.

[SD] "Fast Inference from Transformers via Speculative Decoding", section
"方法细节" (E[#tokens], the acceptance rate alpha = E(beta), the walltime and
operation factors) and its FAQ on choosing gamma (maximise the walltime
factor numerically; a larger cost ratio c gives a smaller optimal gamma; with
alpha > c there is a gain of at least (1 + alpha)/(1 + c); an oracle that
picks gamma per step is bounded by 1/(1 - alpha) tokens per call). The
appendix E worked example (6.86x, 1.6x) is pinned in test_oracle_sps.py.
"""

import numpy as np
import pytest

import oracle


def _tokens_by_law(alpha, gamma):
    """E[#tokens] from the law of the number of accepted drafts (n < gamma:
    alpha^n (1 - alpha); n = gamma: alpha^gamma); n + 1 tokens are emitted."""
    e = 0.0
    for n in range(gamma + 1):
        pn = alpha ** n * (1 - alpha) if n < gamma else alpha ** gamma
        e += pn * (n + 1)
    return e


@pytest.mark.parametrize("alpha", [0.0, 0.2, 0.55, 0.6, 0.8, 0.9, 0.97])
@pytest.mark.parametrize("c", [0.0, 0.01, 0.05, 0.2, 0.5])
def test_best_gamma_by_brute_force(alpha, c):
    gmax = 24
    f = np.array([_tokens_by_law(alpha, g) / (g * c + 1) for g in range(1, gmax + 1)])
    got = oracle.best_gamma(alpha, c, gmax)
    # the chosen length is optimal up to rounding, and no shorter one is
    # better by more than rounding
    assert f[got - 1] >= f.max() - 1e-12
    assert (f[:got - 1] < f[got - 1] + 1e-12).all()


def test_best_gamma_page_properties():
    gmax = 40
    for alpha in (0.3, 0.6, 0.8, 0.9):
        # zero-cost draft: every extra draft token helps (up to the length at
        # which alpha^(gamma+1) is still visible next to 1 in fp64)
        gz = min(gmax, int(np.log(1e-12) / np.log(alpha)) - 1)
        assert oracle.best_gamma(alpha, 0.0, gz) == gz
        # a larger cost ratio gives a smaller (or equal) optimal gamma
        gs = [oracle.best_gamma(alpha, c, gmax) for c in (0.01, 0.02, 0.05, 0.1, 0.2, 0.5)]
        assert gs == sorted(gs, reverse=True)
        for c in (0.01, 0.1, 0.25):
            if alpha > c:
                g = oracle.best_gamma(alpha, c, gmax)
                assert oracle.walltime_factor(alpha, g, c) >= (1 + alpha) / (1 + c) - 1e-12
                assert oracle.walltime_factor(alpha, 1, c) > 1.0
        for g in range(1, gz + 1):
            assert oracle.expected_tokens(alpha, g) < 1.0 / (1.0 - alpha)
        assert oracle.expected_tokens(alpha, gmax) <= 1.0 / (1.0 - alpha)
    # higher acceptance never shortens the optimal draft
    for c in (0.02, 0.1):
        gs = [oracle.best_gamma(a, c, gmax) for a in (0.2, 0.4, 0.6, 0.8, 0.9, 0.95)]
        assert gs == sorted(gs)
    # no gain when the draft costs more than it is accepted
    assert oracle.walltime_factor(0.2, 1, 0.5) < 1.0


def test_acceptance_rate_and_alpha():
    rng = np.random.default_rng(3)
    q = rng.dirichlet(np.ones(50), size=8)
    p = rng.dirichlet(np.ones(50), size=8)
    beta = oracle.acceptance_rate(q, p)
    # sum min(p, q) = 1 - total variation distance
    np.testing.assert_allclose(beta, 1 - 0.5 * np.abs(q - p).sum(axis=1), rtol=1e-12)
    np.testing.assert_allclose(oracle.acceptance_rate(q, q), 1.0, rtol=1e-12)
    disjoint = oracle.acceptance_rate(np.array([0.5, 0.5, 0, 0]), np.array([0, 0, 0.3, 0.7]))
    assert disjoint == 0.0
    assert oracle.estimate_alpha(beta) == pytest.approx(beta.mean(), rel=1e-15)
    # alpha measured from acceptance frequencies converges to the mean beta
    u = rng.random((200000, 8))
    acc = u < beta[None, :]
    assert abs(acc.mean() - oracle.estimate_alpha(beta)) < 5 * np.sqrt(0.25 / acc.size)
