"""GPU parity of the shared-memory row path against the oracle.

spec_verify takes this path for bf16 logits with a top-k / top-p transform
when V is a multiple of 8 and at most about 54000 (a ring of at least two
rows fits in shared memory: three rows up to about 35000) and both logit
tensors start on 16 bytes. The row maximum, the sum, and the logits within
12 octaves of the maximum (counted per distinct bf16 value, and written as
the target row's window list) come from separate warps; the threshold comes
from the counts, or, when the crossing lies deeper or a warp's list
overflows, from the whole row in the fallback kernel; the residual or bonus
draw reads the window list of its target row, or the rows when the list is
incomplete. These cases cover each of those branches, rings of three and
two rows, V beyond the path (65536: the streaming kernel), batches smaller
and larger than the number of CTAs, and bad rows.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_05_gb300 as sv
from parity import assert_linear_parity, assert_probs, np_
from test_gpu_verify import deep_tie_logits, run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V", [8, 24, 1000, 4096, 32000, 32768, 40000, 65536])
@pytest.mark.parametrize("T,top_p,top_k", [(0.8, 0.95, 0), (1.0, 1.0, 40), (0.7, 0.9, 300)])
def test_vocabularies_and_transforms(V, T, top_p, top_k):
    B = 9 if V >= 32000 else 37
    zt, zd = workloads.linear_logits(B, 3, V, 40 + V, dtype="bf16", sd_t=3.0, sd_d=0.7, boost=5.0, boost_p=0.01)
    run(zt, zd, T, top_p, top_k, seed=V % 97, offset=7, label=f"smem V={V} T={T} p={top_p} k={top_k}",
        max_near=0.05)


def test_many_sequences_more_rows_than_sms():
    """4000 sequences of gamma = 4: each CTA cycles its ring buffers many times."""
    zt, zd = workloads.config_logits("nucleus", 61, steps=500, device="cuda")
    c = workloads.CONFIGS["nucleus"]
    drafts = workloads.gumbel_drafts(zd, c["temperature"], 3)
    g = sv.verify(zt, zd, drafts, c["temperature"], c["top_p"], 0, 17, 0, debug=True)
    idx = np.random.default_rng(5).choice(zt.shape[0], 24, replace=False)
    dn = np_(drafts)
    for b in idx:
        r = oracle.verify(zt[b:b + 1].float().cpu().numpy(), zd[b:b + 1].float().cpu().numpy(), dn[b:b + 1],
                          c["temperature"], c["top_p"], 0, 17, int(b))
        gs = {k: v[b:b + 1] for k, v in g.items()}
        assert_linear_parity(gs, r, max_near_frac=0.05, label="smem x500")
        assert_probs(gs["probs"], r, "smem x500")


def test_crossing_below_the_window():
    """The nucleus ends 16 octaves below the maximum: the candidates within
    12 octaves do not reach it and the selection runs over the resident row."""
    zt, zd = deep_tie_logits(10, 2, 40000, 0.5, 31, "bf16")
    g, r, _ = run(zt, zd, 0.5, 0.97, 0, seed=3, label="smem deep tie", max_near=0.05)
    assert (r["accepted"] < 2).any()


def test_flat_rows_many_candidates_and_long_kept_lists():
    """Flat rows: thousands of logits near the maximum (more candidates than
    are compacted) and nuclei of thousands of tokens (longer than a kept
    list, so the draw reads the rows)."""
    zt, zd = workloads.linear_logits(12, 2, 40000, 23, dtype="bf16", sd_t=0.2, sd_d=0.3)
    run(zt, zd, 1.0, 0.9, 0, seed=8, label="smem flat top-p", max_near=0.05)
    run(zt, zd, 1.0, 1.0, 3000, seed=9, label="smem flat top-k", max_near=0.05)


@pytest.mark.parametrize("gamma", [31, 32, 40])
def test_draft_lengths_beyond_one_warp(gamma):
    """gamma at and beyond 32: the acceptance tests run 32 positions a round,
    the bonus row can lie in the second round, and (gamma >= 10) the window
    list sizes of row n are read on their own. Drafts close to the target, so
    that sequences accept past position 32 and some take the bonus; a top-k
    transform, so that no threshold sits on a near-tie of the kept mass (a
    sequence has 2 gamma + 1 rows that could hold one)."""
    zt, zd = workloads.linear_logits(6, gamma, 32000, 70 + gamma, dtype="bf16", sd_t=3.0, sd_d=0.05, boost=5.0,
                                     boost_p=0.01)
    g, r, _ = run(zt, zd, 0.8, 1.0, 300, seed=gamma, label=f"smem gamma={gamma}", max_near=0.0)
    if gamma >= 32:
        assert (r["accepted"] >= 32).any()


def test_ties_top_k_and_top_p():
    g = torch.Generator().manual_seed(5)
    zt = (torch.randint(-6, 7, (16, 4, 3000), generator=g).float() * 0.5).bfloat16()
    zd = (zt[:, :3].float() + 0.5 * torch.randint(-1, 2, (16, 3, 3000), generator=g).float()).bfloat16()
    run(zt, zd, 1.0, 1.0, 10, seed=9, label="smem ties top-k")
    run(zt, zd, 1.0, 0.6, 0, seed=10, label="smem ties top-p")
    run(zt, zd, 1.0, 0.6, 20, seed=11, label="smem ties top-k top-p")


@pytest.mark.parametrize("lenience", [0.3, 0.8])
def test_lenience(lenience):
    zt, zd = workloads.config_logits("nucleus", 1002, steps=6, sd_d=1.5)
    drafts = oracle.sample(zd, 0.8, 0.95, 0, seed=4)["tokens"]
    g = sv.verify(zt.cuda(), zd.cuda(), torch.from_numpy(drafts).int().cuda(), 0.8, 0.95, 0, 2, 0, debug=True,
                  lenience=lenience)
    r = oracle.verify(zt, zd, drafts, 0.8, 0.95, 0, 2, 0, lenience=lenience)
    assert_linear_parity(g, r, max_near_frac=0.05, label=f"smem l={lenience}")
    assert_probs(g["probs"], r, f"smem l={lenience}")


def test_bad_rows():
    zt, zd = workloads.linear_logits(6, 3, 4096, 8, dtype="bf16")
    zt[1, 2, 100] = float("nan")
    zd[2, 0, 5] = float("inf")
    zt[3, 1, :] = float("-inf")          # a row of only -inf
    zt[0, 0, :1000] = float("-inf")      # -inf alone is fine
    drafts = torch.from_numpy(oracle.sample(zd.float().nan_to_num(posinf=0.0), 1.0, 0.9, seed=1)["tokens"]).int()
    drafts[4, 1] = 4096                  # out of range
    drafts[5, 0] = -1
    run(zt, zd, 1.0, 0.9, 0, seed=4, drafts=drafts.numpy(), label="smem bad inputs")
    r = sv.verify(zt.cuda(), zd.cuda(), drafts.cuda(), 1.0, 0.9)
    assert np_(r["status"]).tolist() == [0, 4, 4, 4, 4, 4]
    assert (np_(r["tokens"])[1:] == -1).all()


def test_unaligned_rows_take_the_streaming_path_with_the_same_results():
    """A draft tensor starting 2 bytes past a 16-byte boundary cannot be
    staged; the streaming kernel verifies it instead, to the same results."""
    zt, zd = workloads.linear_logits(20, 4, 32000, 12, dtype="bf16", sd_t=3.0, sd_d=0.5, boost=6.0, boost_p=0.01)
    drafts = oracle.sample(zd, 0.8, 0.95, 0, seed=2)["tokens"]
    zt_c = zt.cuda()
    big = torch.empty(zd.numel() + 8, dtype=torch.bfloat16, device="cuda")
    zd_c = big[1:1 + zd.numel()].view(zd.shape)
    zd_c.copy_(zd)
    d = torch.from_numpy(drafts).int().cuda()
    a = sv.verify(zt_c, zd_c, d, 0.8, 0.95, 0, 5, 0)
    r = oracle.verify(zt, zd, drafts, 0.8, 0.95, 0, 5, 0)
    assert_linear_parity(a, r, max_near_frac=0.05, label="unaligned draft")
