"""Parity at the bench's own launch sizes: each workload's stacked batch in one
call, exactly as bench.py times it; sampled sequences are recomputed by the
oracle one at a time (offset = b, so every Philox counter is the one the
stacked call used) and compared with the same rules as the smaller tests.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_05_gb300 as sv
import workloads
from parity import assert_linear_parity, assert_mentor_alpha, assert_probs, np_

pytestmark = pytest.mark.gpu


def _oracle_rows(fn, idx):
    """Oracle outputs of sequences idx, one call each, stacked along axis 0."""
    parts = [fn(int(b)) for b in idx]
    out = {}
    for k, v in parts[0].items():
        if isinstance(v, np.ndarray) and v.ndim >= 1:
            out[k] = np.concatenate([p[k] for p in parts], axis=0)
    return out


def _take(g, idx):
    return {k: v[torch.as_tensor(idx, device=v.device)] for k, v in g.items() if isinstance(v, torch.Tensor)}


def test_nucleus_1000_steps_in_one_call():
    c = workloads.CONFIGS["nucleus"]
    zt, zd = workloads.config_logits("nucleus", 2024, steps=1000, device="cuda")
    drafts = workloads.gumbel_drafts(zd, c["temperature"], 5)
    g = sv.verify(zt, zd, drafts, c["temperature"], c["top_p"], 0, 11, 0, debug=True)
    idx = np.random.default_rng(0).choice(zt.shape[0], 32, replace=False)
    dn = np_(drafts)

    def one(b):
        return oracle.verify(zt[b:b + 1].float().cpu().numpy(), zd[b:b + 1].float().cpu().numpy(), dn[b:b + 1],
                             c["temperature"], c["top_p"], 0, 11, b)

    r = _oracle_rows(one, idx)
    gs = _take(g, idx)
    assert_linear_parity(gs, r, max_near_frac=0.05, label="nucleus x1000")
    assert_probs(gs["probs"], r, "nucleus x1000")
    assert (np_(g["status"]) == 0).all() and ((np_(g["accepted"]) >= 0) & (np_(g["accepted"]) <= 4)).all()


def test_mentor_12_steps_in_one_call():
    c = workloads.CONFIGS["mentor"]
    zt, zd = workloads.config_logits("mentor", 2024, steps=12, device="cuda")
    drafts = workloads.gumbel_drafts(zd, c["temperature"], 6)
    g = sv.verify_mentor(zt, zd, drafts, c["temperature"], c["kl_bound"], c["iters"], 13, 0, debug=True)
    idx = np.random.default_rng(1).choice(zt.shape[0], 16, replace=False)
    dn = np_(drafts)

    def one(b):
        return oracle.verify_mentor(zt[b:b + 1].cpu().numpy(), zd[b:b + 1].cpu().numpy(), dn[b:b + 1],
                                    c["temperature"], c["kl_bound"], c["iters"], 13, b)

    r = _oracle_rows(one, idx)
    gs = _take(g, idx)
    assert_linear_parity(gs, r, max_near_frac=0.05, label="mentor x12")
    assert_probs(gs["probs"], r, "mentor x12")
    assert_mentor_alpha(gs["alpha"], r, "mentor x12")
    assert ((r["alpha"] > 0) & (r["alpha"] < 1)).any(), "no sampled position reached the solver"


def test_tree_4_steps_in_one_call():
    c = workloads.CONFIGS["tree"]
    B = c["B"] * 4
    z, tok, par, dep = workloads.tree_inputs(B, c["N"], c["V"], 2024, device="cpu")
    g = sv.verify_tree(z.cuda(), tok.cuda(), par.cuda(), dep.cuda(), c["max_depth"])
    idx = np.random.default_rng(2).choice(B, 10, replace=False)
    r = _oracle_rows(lambda b: oracle.verify_tree(z[b:b + 1].numpy(), tok[b:b + 1].numpy(), par[b:b + 1].numpy(),
                                                  dep[b:b + 1].numpy(), c["max_depth"]), idx)
    gs = _take(g, idx)
    for k in ("accept_len", "path_nodes", "tokens", "bonus", "status"):
        np.testing.assert_array_equal(np_(gs[k]), r[k], err_msg=f"tree x4 {k}")


def test_rest_4_steps_in_one_call():
    c = workloads.CONFIGS["rest"]
    B = c["B"] * 4
    cand = workloads.rest_candidates(B, c["C"], c["L"], c["V"], 2024, bases=c["bases"], diverge=c["diverge"])
    root = np.random.default_rng(2024).integers(0, c["V"], B).astype(np.int32)
    t = sv.tree_build(torch.from_numpy(cand).cuda(), torch.from_numpy(root).cuda(), c["V"], c["N"])
    rb = oracle.rest_tree_batch(cand, None, root, c["N"], c["V"])
    for k, ok in (("node_tokens", "tokens"), ("parent", "parent"), ("depth", "depth"), ("n_nodes", "n_nodes"),
                  ("mask", "mask")):
        np.testing.assert_array_equal(np_(t[k]), rb[ok], err_msg=f"rest x4 {k}")
    z = workloads.forced_tree_logits(rb["tokens"], rb["parent"], rb["n_nodes"], c["V"], 2024, sd=c["sd"],
                                     force_p=c["force_p"], device="cuda")
    g = sv.verify_tree(z, t["node_tokens"], t["parent"], t["depth"], c["L"])
    idx = np.random.default_rng(3).choice(B, 10, replace=False)
    r = _oracle_rows(lambda b: oracle.verify_tree(z[b:b + 1].cpu().numpy(), rb["tokens"][b:b + 1],
                                                  rb["parent"][b:b + 1], rb["depth"][b:b + 1], c["L"]), idx)
    gs = _take(g, idx)
    for k in ("accept_len", "path_nodes", "tokens", "bonus", "status"):
        np.testing.assert_array_equal(np_(gs[k]), r[k], err_msg=f"rest x4 {k}")
