"""spec_acceptance_rate against the oracle: beta = sum_x min(q(x), p(x)) for
every target / draft row pair under the verification transforms.

[SD] "Fast Inference from Transformers via Speculative Decoding", section
"方法细节" (接受率精确刻画). beta is a probability, held to the parity
tolerance of probabilities: 1e-5 relative (fp32 sums of at most V terms in
[0, 1]; the kernel's exponentials are within about 2^-22 of the exact ones and
the sums' rounding errors partly cancel). Rows whose top-p crossing is a
near-tie (the oracle's flag) are left out and counted, as in the verification
parity tests.
"""

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_05_gb300 as sv
import workloads
from parity import BETA_RTOL, record

pytestmark = pytest.mark.gpu
RTOL = BETA_RTOL


def _oracle_beta(zt, zd, T, top_k, top_p):
    B, G1, V = zt.shape
    G = G1 - 1
    q, nt_q = oracle.transformed_probs(zt[:, :G].reshape(-1, V), T, top_k, top_p)
    p, nt_p = oracle.transformed_probs(zd.reshape(-1, V), T, top_k, top_p)
    return oracle.acceptance_rate(q, p).reshape(B, G), (nt_q | nt_p).reshape(B, G)


@pytest.mark.parametrize("case", [
    dict(B=6, G=4, V=1000, dtype="f32", T=1.0, k=0, p=1.0),
    dict(B=5, G=3, V=1001, dtype="f32", T=0.7, k=0, p=0.9),        # rows not 16-byte aligned
    dict(B=4, G=4, V=32000, dtype="bf16", T=0.8, k=0, p=0.95, sd_t=3.0, boost=6.0, boost_p=0.01),
    dict(B=3, G=2, V=4099, dtype="bf16", T=1.3, k=20, p=1.0),       # odd V, top-k
    dict(B=2, G=5, V=32128, dtype="f32", T=1.0, k=50, p=0.8),
    dict(B=1, G=1, V=7, dtype="f32", T=2.0, k=0, p=1.0),
])
def test_beta_matches_oracle(case):
    zt, zd = workloads.linear_logits(case["B"], case["G"], case["V"], seed=17, dtype=case["dtype"],
                                     sd_t=case.get("sd_t", 2.0), boost=case.get("boost", 0.0),
                                     boost_p=case.get("boost_p", 0.0))
    r = sv.acceptance_rate(zt.cuda(), zd.cuda(), case["T"], case["p"], case["k"])
    want, near = _oracle_beta(zt.float().numpy(), zd.float().numpy(), case["T"], case["k"], case["p"])
    got = r["beta"].cpu().numpy()
    assert (r["status"].cpu().numpy() == 0).all()
    ok = ~near
    record(f"beta {case['dtype']} V={case['V']} T={case['T']} k={case['k']} p={case['p']}",
           positions=near.size, near_ties=int(near.sum()))
    assert ok.mean() > 0.8
    np.testing.assert_allclose(got[ok], want[ok], rtol=RTOL, atol=0)
    # alpha as the mean of beta
    assert abs(got[ok].mean() - oracle.estimate_alpha(want[ok])) <= RTOL * oracle.estimate_alpha(want[ok])


def test_full_size_batch_sampled_and_properties():
    """The nucleus workload's 1000 stacked steps (8000 sequences): beta in
    [0, 1], identical rows give 1, and sampled pairs match the oracle."""
    zt, zd = workloads.config_logits("nucleus", 5, steps=1000, device="cuda")
    r = sv.acceptance_rate(zt, zd, 0.8, 0.95, 0)
    beta = r["beta"].cpu().numpy()
    assert beta.shape == (8000, 4) and (r["status"].cpu().numpy() == 0).all()
    assert np.isfinite(beta).all() and (beta >= 0).all() and (beta <= 1 + RTOL).all()
    rng = np.random.default_rng(1)
    for b in rng.choice(8000, 6, replace=False):
        want, near = _oracle_beta(zt[b:b + 1].float().cpu().numpy(), zd[b:b + 1].float().cpu().numpy(),
                                  0.8, 0, 0.95)
        ok = ~near[0]
        record("beta nucleus x1000 (sampled)", positions=near[0].size, near_ties=int(near[0].sum()))
        np.testing.assert_allclose(beta[b][ok], want[0][ok], rtol=RTOL, atol=0)
    same = sv.acceptance_rate(zt[:64], zt[:64, :4].contiguous(), 0.8, 0.95, 0)["beta"]
    np.testing.assert_allclose(same.cpu().numpy(), 1.0, rtol=RTOL, atol=0)


def test_bad_rows_and_host_buffers():
    zt, zd = workloads.linear_logits(3, 2, 500, seed=3)
    zt[1, 0, 7] = float("nan")
    r = sv.acceptance_rate(zt, zd, 1.0)                 # host tensors in, host tensors out
    assert r["beta"].device.type == "cpu"
    assert list(r["status"].numpy()) == [0, 4, 0]
    beta = r["beta"].numpy()
    assert np.isnan(beta[1, 0]) and np.isfinite(beta[1, 1])
    want, _ = _oracle_beta(zt.numpy()[[0, 2]], zd.numpy()[[0, 2]], 1.0, 0, 1.0)
    np.testing.assert_allclose(beta[[0, 2]], want, rtol=RTOL, atol=0)
