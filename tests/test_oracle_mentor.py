"""Pins of the oracle's mentor (lossy) verification.

"推测解码的一种最优有损变体", sections "导师解码" and "解决优化问题": the result
law pi_i = p_i r_i + s_i (1 - sum p r) maximises sum p_i r_i subject to a KL
bound D; the solution has r_i = min(1, q_i/(alpha p_i)), s_i proportional to
max(0, q_i/beta - p_i), KL decreasing in alpha (bisection), r_i >=
min(1, q_i/p_i), and KL(q||p) < D means direct acceptance. The exact alpha of
a given row is pinned only through these properties (parity unpinned beyond
them); D = 0 reduces to standard speculative sampling.
"""

import numpy as np
import pytest
from scipy.optimize import brentq

import oracle
from oracle.spec import transformed_probs
from test_oracle_sps import enumerate_law


def _direct_kl(q, p, alpha):
    """KL(q || pi(alpha)) by direct sums and an independent root finder for beta."""
    R = np.maximum(0.0, p - q / alpha).sum()
    rho = q / p
    if R <= 0:
        beta = rho.max()
    else:
        h = lambda b: np.maximum(0.0, q / b - p).sum() - R
        beta = brentq(h, 1.0 - 1e-12, rho.max() * (1 + 1e-12), xtol=1e-15, rtol=1e-15)
    pi = np.minimum(p, q / alpha) + np.maximum(0.0, q / beta - p)
    return float(np.sum(q * np.log(q / pi))), beta, pi


def _rows(seed, n, V, sd=1.5, noise=1.0):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, sd, (n, V))
    zd = zt + rng.normal(0, noise, (n, V))
    return transformed_probs(zt, 1.0)[0], transformed_probs(zd, 1.0)[0]


def test_d_zero_reproduces_standard_speculative_sampling():
    rng = np.random.default_rng(0)
    B, gamma, V = 400, 4, 30
    zt = rng.normal(0, 2, (B, gamma + 1, V))
    zd = zt[:, :gamma] + rng.normal(0, 1.2, (B, gamma, V))
    x = oracle.sample(zd, 1.0, seed=2)["tokens"]
    a = oracle.verify(zt, zd, x, 1.0, seed=2)
    m = oracle.verify_mentor(zt, zd, x, 1.0, kl_bound=0.0, seed=2)
    np.testing.assert_array_equal(a["tokens"], m["tokens"])
    np.testing.assert_array_equal(a["accepted"], m["accepted"])
    decided = np.arange(gamma)[None, :] <= a["accepted"][:, None]
    solved = decided & (m["alpha"] >= 0)
    assert solved.any()
    assert np.all(m["alpha"][solved] == 1.0)


@pytest.mark.parametrize("D", [0.01, 0.1, 0.3])
def test_solution_is_feasible_tight_and_matches_direct_law(D):
    q, p = _rows(1, 40, 150)
    checked = 0
    for i in range(q.shape[0]):
        sol = oracle.mentor_solve(q[i], p[i], D)
        kl0 = float(np.sum(q[i] * np.log(q[i] / p[i])))
        np.testing.assert_allclose(sol["kl0"], kl0, rtol=1e-12)
        if sol["shortcut"]:
            assert kl0 <= D
            continue
        a, b = sol["alpha"], sol["beta"]
        assert 0 < a <= 1
        pi = oracle.mentor_pi(q[i], p[i], a, b)
        np.testing.assert_allclose(pi.sum(), 1.0, atol=1e-12)
        kl_direct, beta_direct, pi_direct = _direct_kl(q[i], p[i], a)
        np.testing.assert_allclose(b, beta_direct, rtol=1e-9)
        np.testing.assert_allclose(pi, pi_direct, atol=1e-12)
        assert kl_direct <= D * (1 + 1e-12)
        if a < 1 and not sol["near"]:
            # the bisection's other end (alpha - 2^-30) is infeasible: alpha is the smallest
            assert _direct_kl(q[i], p[i], a - 2.0 ** -30)[0] > D
        # r >= min(1, q/p): the mentor never accepts less than the standard test
        r = np.minimum(1.0, q[i] / (a * p[i]))
        assert np.all(r >= np.minimum(1.0, q[i] / p[i]))
        checked += 1
    assert checked > 10


def test_kl_decreases_in_alpha_and_vanishes_at_one():
    q, p = _rows(2, 6, 80)
    alphas = np.linspace(0.05, 1.0, 40)
    for i in range(q.shape[0]):
        kls = [_direct_kl(q[i], p[i], a)[0] for a in alphas]
        assert np.all(np.diff(kls) <= 1e-12)
        assert abs(kls[-1]) < 1e-12
        # and the objective sum p r = sum min(p, q/alpha) decreases too
        obj = [np.minimum(p[i], q[i] / a).sum() for a in alphas]
        assert np.all(np.diff(obj) <= 1e-12)


def test_kl_shortcut_accepts_directly():
    q, p = _rows(3, 10, 60, noise=0.3)
    kl0 = np.sum(q * np.log(q / p), axis=1)
    for i in range(q.shape[0]):
        sol = oracle.mentor_solve(q[i], p[i], kl0[i] * 1.01)
        assert sol["shortcut"] and sol["alpha"] == 0
        np.testing.assert_allclose(oracle.mentor_pi(q[i], p[i], 0.0, np.inf), p[i])


def test_grid_search_finds_nothing_better_on_three_tokens():
    """No feasible (r, s) on a grid beats the KKT solution's sum p r."""
    rng = np.random.default_rng(4)
    step = 0.05
    g = np.arange(0, 1 + 1e-9, step)
    R = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    S = np.array([(a, b, 1 - a - b) for a in g for b in g if a + b <= 1 + 1e-9])
    S = np.clip(S, 0, None)
    for trial in range(6):
        q = rng.dirichlet(np.ones(3) * 2)
        p = rng.dirichlet(np.ones(3) * 2)
        kl0 = np.sum(q * np.log(q / p))
        D = kl0 * rng.uniform(0.15, 0.8)
        sol = oracle.mentor_solve(q, p, D)
        assert not sol["shortcut"]
        best_kkt = np.minimum(p, q / sol["alpha"]).sum()
        A = R @ p                                              # [nr]
        pi = (R * p)[:, None, :] + S[None, :, :] * (1 - A)[:, None, None]
        with np.errstate(divide="ignore", invalid="ignore"):
            kl = np.sum(q * np.log(q / pi), axis=2)
        feas = np.nan_to_num(kl, nan=np.inf) <= D
        best_grid = np.max(np.where(feas.any(axis=1), A, -1))
        assert best_grid <= best_kkt + 1e-9
        assert best_grid >= best_kkt - 0.15   # the grid gets close: the test has teeth


@pytest.mark.parametrize("frac,seed", [(0.2, 0), (0.5, 1), (0.8, 2)])
def test_output_law_equals_pi(frac, seed):
    """Exact enumeration (gamma = 1): the emitted token has law pi."""
    rng = np.random.default_rng(seed + 20)
    V = 4
    zt = rng.normal(0, 1.5, (2, V))
    zd = zt[:1] + rng.normal(0, 1.3, (1, V))
    q = transformed_probs(zt[:1], 1.0)[0][0]
    p = transformed_probs(zd, 1.0)[0][0]
    D = frac * float(np.sum(q * np.log(q / p)))
    sol = oracle.mentor_solve(q, p, D)
    assert not sol["shortcut"]
    a, b = sol["alpha"], sol["beta"]
    s = np.maximum(0.0, q / b - p)
    acc_breaks = {(0, x): [min(1.0, q[x] / (a * p[x]))] for x in range(V)}
    w, r, _, _ = enumerate_law(zt, zd, verify_fn=oracle.verify_mentor, kl_bound=D,
                               acc_breaks=acc_breaks, extra_breaks=[np.cumsum(s) / s.sum()])
    law = np.bincount(r["tokens"][:, 0], weights=w, minlength=V)
    np.testing.assert_allclose(law, oracle.mentor_pi(q, p, a, b), atol=1e-12)


def test_alpha_output_codes():
    rng = np.random.default_rng(5)
    B, gamma, V = 200, 3, 40
    zt = rng.normal(0, 2, (B, gamma + 1, V))
    zd = zt[:, :gamma] + rng.normal(0, 1.2, (B, gamma, V))
    x = oracle.sample(zd, 1.0, seed=1)["tokens"]
    m = oracle.verify_mentor(zt, zd, x, 1.0, kl_bound=0.1, seed=1)
    decided = np.arange(gamma)[None, :] <= m["accepted"][:, None]
    decided &= np.arange(gamma)[None, :] < gamma
    a = m["alpha"][decided]
    assert np.all((a == -1) | (a == 0) | ((a > 0) & (a <= 1)))
    assert (a == -1).any() and ((a > 0) & (a <= 1)).any()
    # a larger bound never accepts fewer tokens on the same uniforms
    m2 = oracle.verify_mentor(zt, zd, x, 1.0, kl_bound=0.5, seed=1)
    assert np.all(m2["accepted"] >= m["accepted"])
