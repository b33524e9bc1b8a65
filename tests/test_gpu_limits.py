"""The largest shapes the boundary accepts: V = SPEC_MAX_V and gamma =
SPEC_MAX_GAMMA, against the oracle (same comparison rules as the other
parity tests). Few long rows also take the row kernel's segmented path (a
row split across CTAs, its threshold from the global selection).
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_05_gb300 as sv
import workloads
from parity import assert_linear_parity, assert_probs, in_adm, np_, record

pytestmark = pytest.mark.gpu

MAX_V = 262144
MAX_GAMMA = 255


def _verify(zt, zd, T, top_p=1.0, top_k=0, seed=3, max_near=0.1, label="", drafts=None):
    if drafts is None:
        drafts = workloads.gumbel_drafts(zd, max(T, 1e-3), seed + 1).cpu().numpy() if T > 0 else \
            zd.float().argmax(dim=2).cpu().numpy()
    g = sv.verify(zt.cuda(), zd.cuda(), torch.from_numpy(drafts).int().cuda(), T, top_p, top_k, seed, 0,
                  debug=True)
    r = oracle.verify(zt.float().numpy(), zd.float().numpy() if T > 0 else None, drafts, T, top_p, top_k, seed, 0)
    assert_linear_parity(g, r, max_near_frac=max_near, label=label)
    if T > 0:
        assert_probs(g["probs"], r, label)
    return g, r


def test_max_vocabulary_and_max_draft_length():
    zt, zd = workloads.linear_logits(1, MAX_GAMMA, MAX_V, seed=21, sd_t=2.0, sd_d=0.3)
    g, r = _verify(zt, zd, 1.0, label="V max, gamma max")
    assert np_(g["tokens"]).shape == (1, MAX_GAMMA + 1)


def test_max_vocabulary_top_p_on_few_rows():
    """Three sequences of gamma = 4 at V = SPEC_MAX_V in bf16: few long rows,
    so rows are split into segments and the top-p threshold comes from the
    selection over the whole row."""
    zt, zd = workloads.linear_logits(3, 4, MAX_V, seed=22, dtype="bf16", sd_t=3.0, sd_d=0.5, boost=6.0,
                                     boost_p=0.01)
    _verify(zt, zd, 0.8, top_p=0.95, label="V max top-p", max_near=0.0)
    _verify(zt, zd, 1.0, top_k=1000, label="V max top-k", max_near=0.0)


def test_max_sizes_at_temperature_zero():
    """Drafts equal to the target argmax for 200 positions, then a wrong token:
    exactly 200 are accepted and the 201st token is the target argmax."""
    zt, zd = workloads.linear_logits(1, MAX_GAMMA, MAX_V, seed=23, sd_t=2.0, sd_d=0.05)
    drafts = zt[:, :MAX_GAMMA].argmax(dim=2).numpy().astype(np.int64)
    drafts[0, 200] = (drafts[0, 200] + 1) % MAX_V
    g, r = _verify(zt, zd, 0.0, label="V max, gamma max, T=0", drafts=drafts)
    assert r["accepted"][0] == 200 and np_(g["accepted"])[0] == 200


def test_sample_at_max_vocabulary():
    z, _ = workloads.linear_logits(4, 1, MAX_V, seed=24)
    z = z[:, :1].contiguous()
    g = sv.sample(z.cuda(), 0.9, 0.9, 0, seed=4, offset=0)
    r = oracle.sample(z.numpy(), 0.9, 0.9, 0, seed=4, offset=0)
    ok = ~r["near_tie"]
    gt = np_(g["tokens"])
    record("sample V max", draws=ok.size, near_ties=int((~ok).sum()),
           draws_not_oracle_token=int((ok & (gt != r["tokens"])).sum()))
    hit = in_adm(gt.reshape(-1), r["adm_tokens"].reshape(gt.size, -1)).reshape(gt.shape)
    assert hit[ok].all()
