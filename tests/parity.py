"""Comparison helpers for the GPU parity tests (no verification arithmetic here).

The bar: integer outputs (accepted counts, emitted tokens, tree
paths, argmax indices) match the oracle exactly, except decisions the oracle
flags as near-ties (a uniform within 1e-5 of the acceptance ratio or of a CDF
boundary, a top-p mass within 1e-5 of top_p, a mentor KL within 1e-5 * D of
D), which are excluded and counted; probabilities and the mentor alpha agree
within 1e-5 relative.
"""

import numpy as np
import torch

PROB_RTOL = 1e-5
ALPHA_RTOL = 1e-5   # mentor alpha, relative
BETA_RTOL = 1e-5    # acceptance probabilities beta = sum min(q, p), relative

# Counts of the decisions each parity test excluded or accepted as equally
# valid, by test label (reported at the end of the session by conftest.py).
NEAR_TIES = {}


def record(label, **counts):
    e = NEAR_TIES.setdefault(label, {})
    for k, v in counts.items():
        e[k] = e.get(k, 0) + int(v)


def np_(t):
    return t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def in_adm(tok, adm):
    """tok [N] lies in its row of the admissible sets adm [N, K] (-1 padded)."""
    return ((adm == np.asarray(tok)[:, None]) & (adm >= 0)).any(axis=1)


def assert_linear_parity(g, r, max_near_frac=0.05, label=""):
    """GPU verify / mentor outputs g against the oracle dict r.

    Rows flagged near_tie are excluded (and counted). The emitted prefix and
    the accepted count match exactly; the final drawn token is one of the
    oracle's admissible draws (the tokens a draw returns when its threshold
    moves within the near-tie band; one token unless the threshold sits next
    to a CDF boundary).
    """
    st = np_(g["status"])
    np.testing.assert_array_equal(st, r["status"], err_msg=f"{label} status")
    acc, tok, nxt = np_(g["accepted"]), np_(g["tokens"]), np_(g["next_token"])
    ok = ~r["near_tie"]
    adm = r["adm_tokens"]
    good = r["status"] == 0
    draw_ok = in_adm(nxt, adm) | ~good
    # the emitted tokens: the accepted prefix exactly, then the drawn token
    G1 = tok.shape[1]
    pos = np.arange(G1)[None, :]
    n = np.clip(r["accepted"], 0, G1 - 1)[:, None]
    prefix_ok = np.where(good[:, None] & (pos == n), True, tok == r["tokens"]).all(axis=1)
    last_ok = np.where(good, tok[np.arange(len(acc)), np.clip(r["accepted"], 0, G1 - 1)] == nxt, True)
    bad = ok & ((acc != r["accepted"]) | ~prefix_ok | ~last_ok | ~draw_ok)
    if bad.any():
        i = np.nonzero(bad)[0][:5]
        raise AssertionError(
            f"{label}: {bad.sum()} mismatches outside near-ties (of {len(acc)}); rows {i.tolist()}: "
            f"gpu acc {acc[i].tolist()} ref {r['accepted'][i].tolist()}, "
            f"gpu next {nxt[i].tolist()} ref {r['next_token'][i].tolist()} admissible {adm[i].tolist()}")
    near = int(r["near_tie"].sum())
    multi = ok & good & ((adm >= 0).sum(axis=1) > 1)
    record(label, sequences=len(acc), near_ties=near, draws_with_several_admissible=int(multi.sum()),
           draws_not_oracle_token=int((ok & good & (nxt != r["next_token"])).sum()),
           threshold_near=int(r["prob_near"].any(axis=1).sum()) if "prob_near" in r else 0)
    assert near <= max(2, max_near_frac * len(acc)), f"{label}: {near} near-ties of {len(acc)}"
    return near


def assert_mentor_alpha(g_alpha, r, label=""):
    """Mentor alpha at the decided positions (k <= accepted) of rows without a
    near-tie: the standard-test (-1) and shortcut (0) codes exactly; every
    bisection result within ALPHA_RTOL of the oracle's, except where the
    oracle's admissible range [alpha_lo, alpha_hi] (bisections whose KL
    evaluations are all off by 1e-5 D) is itself wider than ALPHA_RTOL: such
    an alpha is a near-tie, counted and held to that range (widened by
    ALPHA_RTOL)."""
    ga = np_(g_alpha).astype(np.float64)
    gamma = ga.shape[1]
    dec = (np.arange(gamma)[None, :] <= np.minimum(r["accepted"], gamma - 1)[:, None])
    dec &= ~r["near_tie"][:, None] & (r["status"][:, None] == 0) & ~np.isnan(r["alpha"])
    code = dec & (r["alpha"] <= 0)
    np.testing.assert_array_equal(ga[code], r["alpha"][code], err_msg=f"{label} alpha codes")
    sol = dec & (r["alpha"] > 0)
    a, ra, lo, hi = ga[sol], r["alpha"][sol], r["alpha_lo"][sol], r["alpha_hi"][sol]
    wide = (hi - lo) > ALPHA_RTOL * ra
    rel = np.abs(a - ra) / ra
    bad = ~wide & (rel > ALPHA_RTOL)
    assert not bad.any(), (f"{label}: {bad.sum()} of {sol.sum()} alphas off by more than {ALPHA_RTOL} relative "
                           f"(worst {rel[~wide].max():.3g})")
    inside = (a >= lo * (1 - ALPHA_RTOL)) & (a <= hi * (1 + ALPHA_RTOL))
    assert inside[wide].all(), f"{label}: alpha near-ties outside their admissible range"
    record(label, alphas_solved=int(sol.sum()), alpha_near_ties=int(wide.sum()))
    return float(rel[~wide].max()) if (~wide).any() else 0.0


def assert_probs(g_probs, r, label=""):
    """(q(x), p(x)) per position within PROB_RTOL relative (rows without a threshold near-tie)."""
    gp = np_(g_probs)
    sel = (r["status"][:, None] == 0) & ~r.get("prob_near", np.zeros_like(r["q_x"], bool))
    for j, key in enumerate(("q_x", "p_x")):
        a, b = gp[..., j][sel], r[key][sel]
        np.testing.assert_allclose(a, b, rtol=PROB_RTOL, atol=1e-37, err_msg=f"{label} {key}")
