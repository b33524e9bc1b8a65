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


def np_(t):
    return t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def assert_linear_parity(g, r, max_near_frac=0.05, label=""):
    """GPU verify / mentor outputs g against the oracle dict r.

    Rows flagged near_tie are excluded (and counted). Where the oracle offers
    an alternative final token (its uniform sits within the band of one CDF
    boundary), either token is accepted, with the emitted prefix unchanged.
    """
    st = np_(g["status"])
    np.testing.assert_array_equal(st, r["status"], err_msg=f"{label} status")
    acc, tok, nxt = np_(g["accepted"]), np_(g["tokens"]), np_(g["next_token"])
    ok = ~r["near_tie"]
    alt = r.get("alt_token", np.full(len(acc), -1))
    use_alt = (alt >= 0) & (nxt == alt) & (nxt != r["next_token"])
    ref_tok = r["tokens"].copy()
    rows = np.nonzero(use_alt)[0]
    ref_tok[rows, r["accepted"][rows]] = alt[rows]
    ref_next = np.where(use_alt, alt, r["next_token"])
    bad = ok & ((acc != r["accepted"]) | (tok != ref_tok).any(axis=1) | (nxt != ref_next))
    if bad.any():
        i = np.nonzero(bad)[0][:5]
        raise AssertionError(
            f"{label}: {bad.sum()} mismatches outside near-ties (of {len(acc)}); rows {i.tolist()}: "
            f"gpu acc {acc[i].tolist()} ref {r['accepted'][i].tolist()}, "
            f"gpu next {nxt[i].tolist()} ref {r['next_token'][i].tolist()} alt {alt[i].tolist()}")
    near = int(r["near_tie"].sum())
    assert near <= max(2, max_near_frac * len(acc)), f"{label}: {near} near-ties of {len(acc)}"
    return near


def assert_probs(g_probs, r, label=""):
    """(q(x), p(x)) per position within PROB_RTOL relative (rows without a threshold near-tie)."""
    gp = np_(g_probs)
    sel = (r["status"][:, None] == 0) & ~r.get("prob_near", np.zeros_like(r["q_x"], bool))
    for j, key in enumerate(("q_x", "p_x")):
        a, b = gp[..., j][sel], r[key][sel]
        np.testing.assert_allclose(a, b, rtol=PROB_RTOL, atol=1e-37, err_msg=f"{label} {key}")
