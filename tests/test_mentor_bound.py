"""The inequality the mentor kernels' first bisection round rests on, checked
against the definition of KL(alpha).

[Mentor] "推测解码的一种最优有损变体", section "解决优化问题": for a given alpha
the rejected mass R = sum_{rho < alpha} (p - q/alpha) is spread over the
indices with rho >= beta, where beta solves sum_{rho >= beta} (q/beta - p) = R,
and pi_i = q_i/alpha below alpha, p_i between, q_i/beta above.

The kernels place beta in a bucket of ln(rho) (log-width d) and leave that
bucket's indices out of the resampled set: beta~ = Q_U/(R + P_U) over the
indices above the bucket. This is still a feasible redistribution (every
index above the bucket has rho >= beta~), so its KL bounds the true one from
above, by at most Q_b d^2/2 (1 + Q_b/Q_U) for a bucket of q-mass Q_b. The
true KL is computed here from the definition (beta by bisection on the
mass equation, pi by oracle.mentor_pi), not from the oracle's sorted sums.
"""

import numpy as np
import pytest

import oracle


def _probs(rng, V, sd_t, sd_d):
    zt = rng.normal(0.0, sd_t, V)
    zd = zt + rng.normal(0.0, sd_d, V)
    q = np.exp(zt - zt.max())
    p = np.exp(zd - zd.max())
    return q / q.sum(), p / p.sum()


def _kl(q, pi):
    m = q > 0
    return float(np.sum(q[m] * np.log(q[m] / pi[m])))


def _true_beta(q, p, rho, R):
    """beta with sum_{rho >= beta} (q/beta - p) = R, by bisection (the left
    side falls as beta grows)."""
    def g(b):
        u = rho >= b
        return q[u].sum() / b - p[u].sum()
    lo, hi = 1.0, float(rho.max())
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if g(mid) > R:
            lo = mid
        else:
            hi = mid
    return hi


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("delta", [1.0 / 64, 1.0 / 8])
def test_bucketed_beta_bounds_the_kl_from_above(seed, delta):
    rng = np.random.default_rng(seed)
    q, p = _probs(rng, 600, 2.0, 1.2 + 0.3 * seed)
    rho = q / p
    checked = 0
    for alpha in np.arange(1, 64) / 64.0:
        low = rho < alpha
        R = p[low].sum() - q[low].sum() / alpha
        beta = _true_beta(q, p, rho, R)
        kl_true = _kl(q, oracle.mentor_pi(q, p, alpha, beta))
        # the bucket of ln(rho) holding beta: [b d, (b + 1) d)
        b = int(np.floor(np.log(beta) / delta))
        top = np.exp((b + 1) * delta)
        up = rho >= top
        if not up.any():
            continue
        QU, PU = q[up].sum(), p[up].sum()
        beta_b = QU / (R + PU)
        assert beta_b <= top * (1 + 1e-12)        # feasible: every resampled index has rho >= beta~
        pi_b = np.where(low, q / alpha, np.where(up, q / beta_b, p))
        assert abs(pi_b.sum() - 1.0) < 1e-12       # a distribution
        kl_b = _kl(q, pi_b)
        bucket = (rho >= np.exp(b * delta)) & ~up
        QB = q[bucket].sum()
        assert kl_b >= kl_true - 1e-12
        assert kl_b - kl_true <= QB * delta ** 2 / 2 * (1 + QB / QU) + 1e-12
        checked += 1
    assert checked > 40


def test_bound_is_tight_enough_to_matter():
    """With d = 1/64 the excess is a small fraction of the KL change between
    neighbouring grid points, so round 0 rarely leaves a point open."""
    rng = np.random.default_rng(7)
    q, p = _probs(rng, 2000, 2.0, 1.2)
    rho = q / p
    excess, step = [], []
    prev = None
    for alpha in np.arange(8, 64) / 64.0:
        low = rho < alpha
        R = p[low].sum() - q[low].sum() / alpha
        beta = _true_beta(q, p, rho, R)
        kl_true = _kl(q, oracle.mentor_pi(q, p, alpha, beta))
        b = int(np.floor(np.log(beta) * 64))
        up = rho >= np.exp((b + 1) / 64)
        QU, PU = q[up].sum(), p[up].sum()
        pi_b = np.where(low, q / alpha, np.where(up, q / (QU / (R + PU)), p))
        excess.append(_kl(q, pi_b) - kl_true)
        if prev is not None:
            step.append(prev - kl_true)
        prev = kl_true
    assert max(excess) < 0.05 * min(step)
