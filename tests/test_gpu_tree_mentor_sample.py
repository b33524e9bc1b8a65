"""GPU parity of spec_verify_tree, spec_verify_mentor and spec_sample against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from parity import assert_linear_parity, assert_mentor_alpha, assert_probs, in_adm, np_, record

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- tree ----

def _tree_parity(z, tok, par, dep, max_depth, label=""):
    g = sv.verify_tree(z.cuda(), tok.cuda(), par.cuda(), dep.cuda(), max_depth)
    r = oracle.verify_tree(z, tok, par, dep, max_depth)
    for k in ("status", "accept_len", "path_nodes", "tokens", "bonus"):
        np.testing.assert_array_equal(np_(g[k]), r[k], err_msg=f"{label} {k}")
    return g, r


def test_tree_config_full_size():
    """tree: B=16, N=64, V=32016, f32, seeded trie BFS pseudo-sequences."""
    c = workloads.CONFIGS["tree"]
    z, tok, par, dep = workloads.tree_inputs(c["B"], c["N"], c["V"], 1004)
    g, r = _tree_parity(z, tok, par, dep, c["max_depth"], "tree config")
    assert r["accept_len"].max() >= 2


@pytest.mark.parametrize("N,V,dtype", [(1, 50, "f32"), (2, 7, "f32"), (20, 999, "bf16"),
                                       (128, 4001, "f32"), (1024, 64, "f32")])
def test_tree_shapes(N, V, dtype):
    B = 5
    rng = np.random.default_rng(N + V)
    par = np.full((B, N), -1, np.int32)
    dep = np.zeros((B, N), np.int32)
    for i in range(1, N):
        par[:, i] = rng.integers(0, i, B)
        dep[:, i] = dep[np.arange(B), par[:, i]] + 1
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    z = torch.randn(B, N, V, generator=torch.Generator().manual_seed(N))
    am = z.argmax(dim=2).numpy()
    for b in range(B):       # make some nodes accepted
        for i in range(1, N):
            if rng.random() < 0.6:
                tok[b, i] = am[b, par[b, i]]
    if dtype == "bf16":
        z = z.bfloat16()
    md = int(dep.max())
    _tree_parity(z, torch.from_numpy(tok), torch.from_numpy(par), torch.from_numpy(dep), md, f"N={N}")


def test_tree_malformed_and_bad_rows():
    c = workloads.CONFIGS["tree"]
    z, tok, par, dep = workloads.tree_inputs(6, 16, 3000, 7)
    par[1, 5] = 9          # parent after child
    dep[2, 3] += 1         # depth inconsistent
    tok[3, 4] = 3000       # token out of range
    z[4, 7, 11] = float("nan")
    par[5, 0] = 0          # root with a parent
    g, r = _tree_parity(z, tok, par, dep, 6, "malformed")
    assert np_(g["status"]).tolist() == [0, 4, 4, 4, 4, 4]


# -------------------------------------------------------------- mentor ----

def _mentor(zt, zd, D, seed=0, iters=30, label=""):
    zt_o, zd_o = zt.float().numpy(), zd.float().numpy()  # the oracle reads the same values in fp64
    drafts = oracle.sample(zd_o, 1.0, seed=seed + 11)["tokens"]
    g = sv.verify_mentor(zt.cuda(), zd.cuda(), torch.from_numpy(drafts).int().cuda(), 1.0, D, iters,
                         seed, 0, debug=True)
    r = oracle.verify_mentor(zt_o, zd_o, drafts, 1.0, D, iters, seed, 0)
    assert_linear_parity(g, r, max_near_frac=0.05, label=label)
    assert_probs(g["probs"], r, label)
    assert_mentor_alpha(g["alpha"], r, label)
    return g, r, drafts


@pytest.mark.parametrize("D", [0.01, 0.1])
def test_mentor_config_full_size(D):
    """mentor: B=32, gamma=5, V=32128, f32, T=1, 30 bisection steps."""
    zt, zd = workloads.config_logits("mentor", 1005)
    g, r, _ = _mentor(zt, zd, D, seed=2, label=f"mentor D={D}")
    solved = (r["alpha"] > 0) & (r["alpha"] < 1)
    assert solved.any()


def test_mentor_bound_zero_equals_standard_verification():
    zt, zd = workloads.linear_logits(24, 4, 6000, 3, sd_t=2.0, sd_d=1.2)
    drafts = torch.from_numpy(oracle.sample(zd, 1.0, seed=5)["tokens"]).int().cuda()
    m = sv.verify_mentor(zt.cuda(), zd.cuda(), drafts, 1.0, 0.0, 30, 9, 0)
    v = sv.verify(zt.cuda(), zd.cuda(), drafts, 1.0, 1.0, 0, 9, 0)
    for k in ("accepted", "tokens", "next_token", "status"):
        np.testing.assert_array_equal(np_(m[k]), np_(v[k]))


@pytest.mark.parametrize("V,iters", [(3, 30), (100, 30), (5000, 12), (40001, 30), (40000, 30), (262144, 30)])
def test_mentor_shapes(V, iters):
    """Small and odd vocabularies; above 32768 entries the pass-1 bucket ids
    live in global scratch (40001: scalar accesses, 40000: 16-byte ones);
    262144 is the largest vocabulary the boundary accepts."""
    zt, zd = workloads.linear_logits(12, 3, V, V, sd_t=2.0, sd_d=1.2)
    _mentor(zt, zd, 0.05, seed=V, iters=iters, label=f"mentor V={V}")


@pytest.mark.parametrize("iters", [1, 5, 10, 40, 64])
def test_mentor_bisection_depths(iters):
    """Up to ten levels the first round alone decides; beyond 2^-60 levels
    change alpha by less than any tolerance and are not taken."""
    zt, zd = workloads.linear_logits(10, 3, 4099, 7 + iters, sd_t=2.0, sd_d=1.2)
    _mentor(zt, zd, 0.05, seed=iters, iters=iters, label=f"iters={iters}")


def test_mentor_loose_bound_and_extreme_rows():
    """A loose bound on far-apart rows (results below 2^-10 with levels left:
    the sorting solve takes those rows), then peaked targets with
    zero-probability logits on either side (q > 0 = p makes KL(q || p)
    infinite and rho infinite)."""
    zt, zd = workloads.linear_logits(12, 3, 3000, 21, sd_t=2.0, sd_d=4.0)
    _, r, _ = _mentor(zt, zd, 2.0, seed=3, label="loose bound")
    assert ((r["alpha"] > 0) & (r["alpha"] < 2.0 ** -10)).any(), "no row took a result below 2^-10"
    zt2, zd2 = workloads.linear_logits(12, 3, 3000, 22, sd_t=6.0, sd_d=1.0)
    zt2[:, :, 5] += 12.0
    zd2[:, :, 3::7] = float("-inf")
    zt2[:, :, 1::11] = float("-inf")
    _mentor(zt2, zd2, 0.1, seed=4, label="extremes")


def test_mentor_bf16():
    zt, zd = workloads.linear_logits(10, 3, 32000, 31, dtype="bf16", sd_t=2.0, sd_d=1.2)
    _, r, _ = _mentor(zt, zd, 0.1, seed=1, label="mentor bf16")
    assert ((r["alpha"] > 0) & (r["alpha"] < 1)).any()


# -------------------------------------------------------------- sample ----

@pytest.mark.parametrize("dtype,T,top_p,top_k", [("f32", 1.0, 1.0, 0), ("bf16", 0.8, 0.95, 0),
                                                 ("f32", 0.0, 1.0, 0), ("f32", 1.2, 0.9, 40),
                                                 ("bf16", 0.0, 1.0, 0)])
def test_sample_matches_oracle(dtype, T, top_p, top_k):
    zt, _ = workloads.linear_logits(20, 3, 32000, 13, dtype=dtype, sd_t=3.0)
    g = sv.sample(zt.cuda(), T, top_p, top_k, seed=4, offset=100, pos0=2)
    r = oracle.sample(zt, T, top_p, top_k, seed=4, offset=100, pos0=2)
    ok = ~r["near_tie"]
    gt = np_(g["tokens"])
    hit = in_adm(gt.reshape(-1), r["adm_tokens"].reshape(gt.size, -1)).reshape(gt.shape)
    record(f"sample {dtype} T={T} p={top_p} k={top_k}", draws=ok.size, near_ties=int((~ok).sum()),
           draws_not_oracle_token=int((ok & (gt != r["tokens"])).sum()))
    assert hit[ok].all(), np.nonzero(~hit & ok)
    np.testing.assert_array_equal(np_(g["status"]), r["status"])
