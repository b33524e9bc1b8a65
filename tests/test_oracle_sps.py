"""Pins of the oracle's modified rejection sampling against what the pages fix.

* Theorem 1 ("Accelerating Large Language Model Decoding with Speculative
  Sampling", appendix proof): the emitted token has law q. Checked exactly by
  integrating every uniform over the cells between the decision boundaries,
  and by a chi-square test over 10^6 seeded trials at V=8.
* Rejection probability sum max(0, q-p) = 1 - sum min(p, q) (same proof) and
  alpha = 1 - E[D_LK] ("Fast Inference from Transformers via Speculative
  Decoding" write-up, "接受率精确刻画").
* E[#tokens] = (1 - alpha^(gamma+1))/(1 - alpha) (same write-up,
  "期望生成 token 数"), exact under i.i.d. acceptance.
* The appendix E worked example (6.86x speedup at 1.6x operations).
"""

import itertools
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from oracle import PURPOSE_ACCEPT, PURPOSE_RESAMPLE, PURPOSE_DRAFT
from oracle.spec import transformed_probs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cells(breaks):
    b = np.unique(np.clip(np.asarray(breaks, dtype=np.float64), 0.0, 1.0))
    b = np.union1d(b, [0.0, 1.0])
    lo, hi = b[:-1], b[1:]
    keep = hi > lo
    return 0.5 * (lo[keep] + hi[keep]), (hi - lo)[keep]


def enumerate_law(zt, zd, temperature=1.0, top_p=1.0, top_k=0, verify_fn=None, **kw):
    """Run the oracle on every (drafts, uniform-cell) branch of one sequence.

    Each uniform ranges over the cells between the decision boundaries (the
    acceptance threshold min(1, q/p) and the cumulative residual / bonus
    masses). Every branch is evaluated at the cell midpoints and, one uniform
    at a time, just inside both ends of its cell; the oracle's output must be
    the same at all probes (so its boundaries sit where the pages put them),
    and the midpoint runs carry the exact branch probabilities:
    prod p_k(x_k) times the cell lengths. Returns (weights, result, q, p) for
    the midpoint runs.
    """
    verify_fn = verify_fn or oracle.verify
    G1, V = zt.shape
    g = G1 - 1
    q = [transformed_probs(zt[k:k + 1], temperature, top_k, top_p)[0][0] for k in range(G1)]
    p = [transformed_probs(zd[k:k + 1], temperature, top_k, top_p)[0][0] for k in range(g)]
    res_breaks = [0.0, 1.0]
    for k in range(g):
        w = np.maximum(0.0, q[k] - p[k])
        w = w if w.sum() > 0 else q[k]
        res_breaks += list(np.cumsum(w) / w.sum())
    res_breaks += list(np.cumsum(q[g]) / q[g].sum())
    for extra in kw.pop("extra_breaks", []):
        res_breaks += list(extra)
    acc_breaks = kw.pop("acc_breaks", {})
    res_mid, res_len = _cells(res_breaks)
    eps = 1e-9

    base = []   # (x, acc (mid, len) per position, res (mid, len))
    for x in itertools.product(range(V), repeat=g):
        px = np.prod([p[k][x[k]] for k in range(g)]) if g else 1.0
        if px == 0:
            continue
        acc_cells = []
        for k in range(g):
            thr = min(1.0, q[k][x[k]] / p[k][x[k]])
            acc_cells.append(_cells([thr] + list(acc_breaks.get((k, x[k]), []))))
        for choice in itertools.product(*[range(len(c[0])) for c in acc_cells]):
            acc = [(acc_cells[k][0][c], acc_cells[k][1][c]) for k, c in enumerate(choice)]
            for j in range(len(res_mid)):
                base.append((x, acc, (res_mid[j], res_len[j]), px))
    xs, ua, ur, wt, grp = [], [], [], [], []
    for gi, (x, acc, res, px) in enumerate(base):
        mids = [a[0] for a in acc] + [res[0]]
        lens = [a[1] for a in acc] + [res[1]]
        variants = [(mids, px * np.prod(lens))]
        for j in range(g + 1):
            d = min(eps, lens[j] / 4)
            for v in (mids[j] - lens[j] / 2 + d, mids[j] + lens[j] / 2 - d):
                m2 = list(mids)
                m2[j] = v
                variants.append((m2, 0.0))
        for m2, wgt in variants:
            xs.append(x)
            ua.append(m2[:g])
            ur.append(m2[g])
            wt.append(wgt)
            grp.append(gi)
    M = len(wt)
    ua = np.asarray(ua, dtype=np.float64).reshape(M, g)
    ur = np.asarray(ur)

    def ufn(rows, pos, purpose):
        idx = np.asarray(rows, dtype=np.int64)
        if purpose == PURPOSE_ACCEPT:
            return ua[idx, pos]
        return ur[idx]

    tt = np.broadcast_to(zt, (M, G1, V))
    dd = np.broadcast_to(zd, (M, g, V))
    extra = {"top_p": top_p, "top_k": top_k} if verify_fn is oracle.verify else {}
    r = verify_fn(tt, dd, np.asarray(xs, dtype=np.int64).reshape(M, g), temperature=temperature,
                  uniform_fn=ufn, **extra, **kw)
    grp = np.asarray(grp)
    wt = np.asarray(wt)
    first = np.r_[True, grp[1:] != grp[:-1]]
    head = np.nonzero(first)[0]
    same = (r["tokens"] == r["tokens"][head[grp]]).all(axis=1)
    assert same.all(), "oracle output changes inside a decision cell"
    sel = first
    out = {k: (v[sel] if isinstance(v, np.ndarray) and v.shape[:1] == (M,) else v) for k, v in r.items()}
    return wt[sel], out, q, p


CASES = [
    # (V, gamma, T, top_p, top_k, seed)
    (2, 1, 1.0, 1.0, 0, 0),
    (3, 1, 0.7, 1.0, 0, 1),
    (4, 2, 1.0, 1.0, 0, 2),
    (5, 1, 1.3, 1.0, 0, 3),
    (5, 2, 0.8, 0.9, 0, 4),
    (5, 2, 1.0, 1.0, 3, 5),
    (4, 3, 1.0, 0.8, 3, 6),
]


@pytest.mark.parametrize("V,gamma,T,top_p,top_k,seed", CASES)
def test_theorem1_exact_enumeration(V, gamma, T, top_p, top_k, seed):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, (gamma + 1, V))
    zd = zt[:gamma] + rng.normal(0, 1.0, (gamma, V))
    w, r, q, p = enumerate_law(zt, zd, T, top_p, top_k)
    assert abs(w.sum() - 1.0) < 1e-12
    tok = r["tokens"]
    # first emitted token ~ q_0 (Theorem 1)
    law0 = np.bincount(tok[:, 0], weights=w, minlength=V)
    np.testing.assert_allclose(law0, q[0], atol=1e-12)
    # given the first token was an accepted draft, the next token ~ q_1
    if gamma >= 2:
        acc0 = r["accepted"] >= 1
        for a in range(V):
            sel = acc0 & (tok[:, 0] == a)
            if w[sel].sum() < 1e-9:
                continue
            law1 = np.bincount(tok[sel, 1], weights=w[sel], minlength=V) / w[sel].sum()
            np.testing.assert_allclose(law1, q[1], atol=1e-10)
    # P(reject at position 0) = sum max(0, q0 - p0) = 1 - sum min(p0, q0)
    rej0 = w[r["accepted"] == 0].sum()
    np.testing.assert_allclose(rej0, np.maximum(0, q[0] - p[0]).sum(), atol=1e-12)
    np.testing.assert_allclose(rej0, 1 - oracle.acceptance_rate(q[0], p[0]), atol=1e-12)


@pytest.mark.parametrize("gamma", [1, 2, 3])
def test_expected_tokens_exact(gamma):
    rng = np.random.default_rng(10 + gamma)
    V = 4
    row_t = rng.normal(0, 1.0, V)
    row_d = row_t + rng.normal(0, 0.8, V)
    zt = np.tile(row_t, (gamma + 1, 1))
    zd = np.tile(row_d, (gamma, 1))
    w, r, q, p = enumerate_law(zt, zd)
    alpha = oracle.acceptance_rate(q[0], p[0])
    emitted = (r["accepted"] + 1).astype(np.float64)
    np.testing.assert_allclose((w * emitted).sum(), oracle.expected_tokens(alpha, gamma), rtol=1e-12)


def test_alpha_is_one_minus_total_variation():
    rng = np.random.default_rng(3)
    q = rng.dirichlet(np.ones(50), size=20)
    p = rng.dirichlet(np.ones(50), size=20)
    d_lk = 0.5 * np.abs(q - p).sum(axis=1)
    np.testing.assert_allclose(oracle.acceptance_rate(q, p), 1 - d_lk, atol=1e-14)
    np.testing.assert_allclose(oracle.acceptance_rate(q, q), 1.0, atol=1e-14)


def test_chi_square_one_million_trials():
    """10^6 seeded trials at V=8, gamma=2: emitted tokens follow q."""
    V, gamma, n = 8, 2, 1_000_000
    rng = np.random.default_rng(99)
    zt = rng.normal(0, 1.2, (gamma + 1, V))
    zd = zt[:gamma] + rng.normal(0, 0.9, (gamma, V))
    tt = np.broadcast_to(zt, (n, gamma + 1, V))
    dd = np.broadcast_to(zd, (n, gamma, V))
    drafts = oracle.sample(dd, 1.0, seed=5)["tokens"]
    r = oracle.verify(tt, dd, drafts, 1.0, seed=5)
    q0 = transformed_probs(zt[:1], 1.0)[0][0]
    q1 = transformed_probs(zt[1:2], 1.0)[0][0]
    p0 = transformed_probs(zd[:1], 1.0)[0][0]
    c0 = np.bincount(r["tokens"][:, 0], minlength=V)
    assert stats.chisquare(c0, q0 * n).pvalue > 1e-3
    sel = r["accepted"] >= 1
    c1 = np.bincount(r["tokens"][sel, 1], minlength=V)
    assert stats.chisquare(c1, q1 * sel.sum()).pvalue > 1e-3
    # acceptance frequency at position 0 -> sum min(p, q)
    beta = oracle.acceptance_rate(q0, p0)
    se = np.sqrt(beta * (1 - beta) / n)
    assert abs(sel.mean() - beta) < 5 * se
    # the draft sampler itself follows p
    assert stats.chisquare(np.bincount(drafts[:, 0], minlength=V), p0 * n).pvalue > 1e-3


def test_expected_tokens_monte_carlo():
    V, gamma, n = 6, 4, 200_000
    rng = np.random.default_rng(17)
    row_t = rng.normal(0, 1.0, V)
    row_d = row_t + rng.normal(0, 0.7, V)
    tt = np.broadcast_to(row_t, (n, gamma + 1, V))
    dd = np.broadcast_to(row_d, (n, gamma, V))
    drafts = oracle.sample(dd, 1.0, seed=3)["tokens"]
    r = oracle.verify(tt, dd, drafts, 1.0, seed=3)
    q = transformed_probs(row_t[None], 1.0)[0][0]
    p = transformed_probs(row_d[None], 1.0)[0][0]
    alpha = oracle.acceptance_rate(q, p)
    emitted = r["accepted"] + 1
    assert abs(emitted.mean() - oracle.expected_tokens(alpha, gamma)) < 5 * emitted.std() / np.sqrt(n)


def test_draft_token_with_zero_draft_probability():
    """p(x) = 0: rho = +inf accepts when q(x) > 0, rho = 0 rejects when q(x) = 0."""
    zt = np.array([[0.0, 1.0, 2.0, 3.0], [0.0, 0.0, 0.0, 0.0]])
    zd = np.array([[5.0, 0.0, 0.0, 0.0]])
    # top_k=1 makes p one-hot at index 0; x=3 has p=0 and q>0 -> always accepted
    r = oracle.verify(zt[None], zd[None], np.array([[3]]), 1.0, top_k=1, seed=0)
    # with top_k=1 the target keeps only index 3, so q(3)=1 and the bonus row is uniform
    assert r["accepted"][0] == 1 and r["tokens"][0, 0] == 3
    r = oracle.verify(zt[None], zd[None], np.array([[1]]), 1.0, top_k=1, seed=0)
    # x=1: q(1)=0 (outside the target's top-1) and p(1)=0 -> rejected, resampled token is 3
    assert r["accepted"][0] == 0 and r["tokens"][0, 0] == 3


def test_temperature_zero_is_the_low_temperature_limit():
    rng = np.random.default_rng(4)
    B, gamma, V = 300, 3, 50
    zt = rng.normal(0, 1, (B, gamma + 1, V))
    zd = zt[:, :gamma] + rng.normal(0, 0.3, (B, gamma, V))
    x = np.argmax(zd, axis=2)
    r0 = oracle.verify(zt, None, x, 0.0)
    r_small = oracle.verify(zt, zd, x, 1e-4, seed=8)
    np.testing.assert_array_equal(r0["accepted"], r_small["accepted"])
    np.testing.assert_array_equal(r0["tokens"], r_small["tokens"])
    # and it is greedy decoding: accept while x_k = argmax, emit the argmax
    am = np.argmax(zt, axis=2)
    for b in range(B):
        n = 0
        while n < gamma and x[b, n] == am[b, n]:
            n += 1
        assert r0["accepted"][b] == n and r0["next_token"][b] == am[b, n]


def test_bad_rows_give_status_and_no_tokens():
    rng = np.random.default_rng(5)
    zt = rng.normal(0, 1, (4, 3, 10))
    zd = rng.normal(0, 1, (4, 2, 10))
    zt[1, 2, 3] = np.nan
    zd[2, 0, 0] = np.inf
    x = np.zeros((4, 2), np.int64)
    x[3, 1] = 10
    zt[0, 0, :] = -np.inf
    zt[0, 0, 4] = 1.0          # -inf alone is allowed
    r = oracle.verify(zt, zd, x, 1.0)
    assert list(r["status"]) == [0, 4, 4, 4]
    assert (r["tokens"][1:] == -1).all() and (r["accepted"][1:] == -1).all()
    zt[0, 1, :] = -np.inf      # a row of only -inf is an error
    assert oracle.verify(zt, zd, x, 1.0)["status"][0] == 4


def test_worked_example_speedup_and_operations():
    with open(os.path.join(GOLDEN, "sd_appendix_e_worked_example.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for a, g, c, ch, wf, of in rows:
        a, g, c, ch = float(a), int(g), float(c), float(ch)
        assert round(oracle.walltime_factor(a, g, c), 2) == float(wf)
        assert round(oracle.ops_factor(a, g, ch), 1) == float(of)
    assert oracle.expected_tokens(1.0, 7) == 8.0


def test_admissible_draws_match_brute_force_threshold_moves():
    """admissible_draws lists exactly the indices inverse_cdf returns when
    its threshold u W moves anywhere within +-NEAR_TIE W (brute force over a
    fine grid of moved uniforms), and always contains the unmoved draw."""
    from oracle.spec import NEAR_TIE, admissible_draws, inverse_cdf

    rng = np.random.default_rng(7)
    for trial in range(300):
        V = int(rng.integers(1, 9))
        w = rng.random((1, V)) * (rng.random((1, V)) < 0.7)
        if trial % 3 == 0:
            w *= 1e-6 * (rng.random((1, V)) < 0.5) + 1.0  # weights next to the band's width
        if w.sum() == 0:
            w[0, 0] = 1.0
        W = w.sum()
        u = float(rng.random())
        if trial % 5 == 0:  # put the threshold right on a boundary
            u = float(np.cumsum(w)[rng.integers(0, V)] / W)
        adm, over = admissible_draws(np.array([u]), w)
        assert not over[0]
        got = set(adm[0][adm[0] >= 0].tolist())
        i0 = int(inverse_cdf(np.array([u]), w)[0][0])
        assert i0 in got
        want = set()
        for du in np.linspace(-NEAR_TIE, NEAR_TIE, 4001):
            uu = max(u + du, 0.0)  # a uniform is never negative
            t = uu * W
            C = np.cumsum(w[0])
            j = int(np.argmax(C > t)) if (C > t).any() else int(np.nonzero(w[0] > 0)[0][-1])
            want.add(j)
        # the grid can miss an interval narrower than its step, never add one
        assert want <= got
        step = 2 * NEAR_TIE * W / 4000
        for j in got - want:
            lo = np.cumsum(w[0])[j] - w[0, j]
            assert w[0, j] <= 2 * step or abs(lo - u * W) >= NEAR_TIE * W - 2 * step \
                or abs(np.cumsum(w[0])[j] - u * W) >= NEAR_TIE * W - 2 * step
