"""Distribution of the GPU path's emitted tokens (Theorem 1 of the speculative
sampling notes, "改进的拒绝采样" and its appendix proof): whatever the draft,
the first emitted token follows q, the next one follows q given acceptance,
and position 0 accepts with probability sum_x min(p(x), q(x)).

10^6 seeded trials at V = 8, gamma = 2, drafts from the library's own sampler,
verified in one call; the expected laws come from the transformed softmax of
the fixed rows (fp64). Chi-square with 7 degrees of freedom, p-value > 1e-3.
"""

import numpy as np
import pytest
import torch

scipy_stats = pytest.importorskip("scipy.stats")

import oracle
import speculative_decoding_verification_05_gb300 as sv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,top_p,top_k", [(1.0, 1.0, 0), (0.8, 0.9, 0), (1.3, 1.0, 5)])
def test_emitted_tokens_follow_the_target_law(T, top_p, top_k):
    V, gamma, n = 8, 2, 1_000_000
    rng = np.random.default_rng(99)
    zt = rng.normal(0, 1.2, (gamma + 1, V))
    zd = zt[:gamma] + rng.normal(0, 0.9, (gamma, V))
    tt = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zt, (n, gamma + 1, V)))).float().cuda()
    dd = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zd, (n, gamma, V)))).float().cuda()
    drafts = sv.sample(dd, T, top_p, top_k, seed=5, purpose=sv.PURPOSE_DRAFT)["tokens"]
    r = sv.verify(tt, dd, drafts, T, top_p, top_k, seed=5)
    tok = r["tokens"].cpu().numpy()
    acc = r["accepted"].cpu().numpy()
    assert (r["status"].cpu().numpy() == 0).all()
    q = oracle.transformed_probs(zt.astype(np.float32), T, top_k, top_p)[0]
    p = oracle.transformed_probs(zd.astype(np.float32), T, top_k, top_p)[0]
    # the draft sampler follows p
    c = np.bincount(drafts[:, 0].cpu().numpy(), minlength=V)
    keep = p[0] > 0
    assert c[~keep].sum() == 0
    assert scipy_stats.chisquare(c[keep], p[0][keep] * n).pvalue > 1e-3
    # the first emitted token follows q_0
    c0 = np.bincount(tok[:, 0], minlength=V)
    keep = q[0] > 0
    assert c0[~keep].sum() == 0
    assert scipy_stats.chisquare(c0[keep], q[0][keep] * n).pvalue > 1e-3
    # given position 0 accepted, the second token follows q_1
    sel = acc >= 1
    c1 = np.bincount(tok[sel, 1], minlength=V)
    keep = q[1] > 0
    assert c1[~keep].sum() == 0
    assert scipy_stats.chisquare(c1[keep], q[1][keep] * sel.sum()).pvalue > 1e-3
    # acceptance frequency at position 0 -> sum_x min(p, q)
    beta = oracle.acceptance_rate(q[0], p[0])
    se = np.sqrt(beta * (1 - beta) / n)
    assert abs(sel.mean() - beta) < 5 * se
