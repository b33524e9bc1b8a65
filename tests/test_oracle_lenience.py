"""Pins for the oracle's lenient verification ([SD] "方法细节", the lenience
extension of its appendix F: the draft probability is scaled by l before the
comparison; no token is emitted with probability above q(x)/l).

* l = 1 reproduces exact verification.
* Exact enumeration over every branch of one sequence: the first emitted
  token has the law min(p, q/l) + (1 - sum min(p, q/l)) norm(max(0, q - l p)),
  which never exceeds q/l (the pages' guarantee), and position 0 accepts with
  probability sum min(p, q/l).
"""

import numpy as np
import pytest

import oracle
from oracle import transformed_probs
from test_oracle_sps import enumerate_law


def test_lenience_one_is_exact_verification():
    rng = np.random.default_rng(5)
    zt = rng.normal(0, 2.0, (64, 4, 50))
    zd = zt[:, :3] + rng.normal(0, 0.8, (64, 3, 50))
    drafts = oracle.sample(zd, 0.9, 0.95, 0, seed=2)["tokens"]
    a = oracle.verify(zt, zd, drafts, 0.9, 0.95, 0, seed=7, offset=3)
    b = oracle.verify(zt, zd, drafts, 0.9, 0.95, 0, seed=7, offset=3, lenience=1.0)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def _lenient_law(q, p, l):
    acc = np.minimum(p, q / l)
    w = np.maximum(0.0, q - l * p)
    r = w / w.sum() if w.sum() > 0 else q
    return acc + (1.0 - acc.sum()) * r, acc.sum()


@pytest.mark.parametrize("l", [0.2, 0.5, 0.9])
@pytest.mark.parametrize("V,seed", [(3, 1), (5, 2)])
def test_lenient_law_by_exact_enumeration(l, V, seed):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.3, (2, V))
    zd = zt[:1] + rng.normal(0, 1.0, (1, V))
    q = transformed_probs(zt[:1], 1.0)[0][0]
    p = transformed_probs(zd, 1.0)[0][0]
    # the lenient decision boundaries: acceptance min(1, q/(l p)), residual max(0, q - l p)
    acc_breaks = {(0, x): [min(1.0, q[x] / (l * p[x]))] for x in range(V) if p[x] > 0}
    w = np.maximum(0.0, q - l * p)
    extra = [np.cumsum(w) / w.sum()] if w.sum() > 0 else []
    fn = lambda *a, **k: oracle.verify(*a, lenience=l, **k)
    wt, res, _, _ = enumerate_law(zt, zd, verify_fn=fn, acc_breaks=acc_breaks, extra_breaks=extra)
    first = res["tokens"][:, 0]
    law = np.array([wt[first == x].sum() for x in range(V)])
    want, beta = _lenient_law(q, p, l)
    np.testing.assert_allclose(law.sum(), 1.0, atol=1e-12)
    np.testing.assert_allclose(law, want, atol=1e-12)
    assert np.all(law <= q / l + 1e-12)
    np.testing.assert_allclose(wt[res["accepted"] >= 1].sum(), beta, atol=1e-12)
    if l < 1:  # strictly lenient: the law moves towards p
        assert np.abs(law - q).sum() > 1e-6
