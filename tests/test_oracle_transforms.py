"""Pins of the oracle's sampling transforms.

The transforms come from "Accelerating Large Language Model Decoding with
Speculative Sampling" notes, "与标准采样方法的兼容性" (nucleus, top-k and
temperature are applied to the probabilities before the scheme) and the
"Fast Inference from Transformers via Speculative Decoding" write-up,
"标准化采样框架" (argmax, top-k, nucleus, temperature are all standard
sampling from an adjusted distribution).
"""

import numpy as np
import pytest
from scipy.special import softmax

from oracle.spec import transformed_probs


def test_plain_temperature_is_softmax():
    rng = np.random.default_rng(0)
    z = rng.normal(0, 3, (20, 300))
    for T in (0.5, 1.0, 2.0):
        q, near = transformed_probs(z, T)
        np.testing.assert_allclose(q, softmax(z / T, axis=1), rtol=1e-12, atol=1e-300)
        assert not near.any()


def test_temperature_zero_and_its_limit():
    rng = np.random.default_rng(1)
    z = rng.normal(0, 1, (50, 40))
    z[np.arange(50), np.argmax(z, axis=1)] += 0.05   # a clear argmax in every row
    q0, _ = transformed_probs(z, 0.0)
    assert (q0.sum(axis=1) == 1).all()
    np.testing.assert_array_equal(np.argmax(q0, axis=1), np.argmax(z, axis=1))
    q_small, _ = transformed_probs(z, 1e-3)
    np.testing.assert_allclose(q_small, q0, atol=1e-6)
    # ties: the lowest index wins
    zt = np.array([[1.0, 3.0, 3.0, 0.0]])
    assert transformed_probs(zt, 0.0)[0][0, 1] == 1.0


def test_top_k_one_is_argmax_without_ties():
    rng = np.random.default_rng(2)
    z = rng.normal(0, 1, (30, 25))
    q, _ = transformed_probs(z, 0.7, top_k=1)
    np.testing.assert_array_equal(q, transformed_probs(z, 0.0)[0])


def test_hand_worked_nucleus_example():
    # probabilities 0.5, 0.3, 0.15, 0.05 at T=1; top_p = 0.75 keeps {0.5, 0.3}
    z = np.log(np.array([[0.5, 0.3, 0.15, 0.05]]))
    q, near = transformed_probs(z, 1.0, top_p=0.75)
    np.testing.assert_allclose(q[0], [0.625, 0.375, 0.0, 0.0], rtol=1e-12)
    assert not near[0]
    # the crossing value is kept: top_p = 0.81 needs the third token too
    q, _ = transformed_probs(z, 1.0, top_p=0.81)
    np.testing.assert_allclose(q[0], np.array([0.5, 0.3, 0.15, 0.0]) / 0.95, rtol=1e-12)
    # a tiny top_p keeps only the argmax
    q, _ = transformed_probs(z, 1.0, top_p=1e-6)
    np.testing.assert_allclose(q[0], [1, 0, 0, 0])


def test_hand_worked_ties_and_order():
    z = np.array([[2.0, 1.0, 1.0, 0.0, -1.0]])
    # top-k is tie-inclusive: the 2nd largest value is 1.0, both copies stay
    q, _ = transformed_probs(z, 1.0, top_k=2)
    assert (q[0] > 0).tolist() == [True, True, True, False, False]
    # top-p keeps a whole tie group: 2.0 alone has mass e^2/(e^2+2e) ~ 0.576
    q, _ = transformed_probs(z, 1.0, top_k=3, top_p=0.6)
    assert (q[0] > 0).tolist() == [True, True, True, False, False]
    # top-k first, then top-p on the renormalised top-k distribution
    w = np.exp(z[0, :3])
    frac_first = w[0] / w.sum()
    q, _ = transformed_probs(z, 1.0, top_k=3, top_p=frac_first - 1e-3)
    assert (q[0] > 0).tolist() == [True, False, False, False, False]


def _brute_force_keep(z, T, top_k, top_p):
    """O(V^2) definition: thresholds by direct sums over the row."""
    V = z.size
    keep = np.ones(V, bool)
    if 0 < top_k < V:
        kth = max(v for v in z if np.sum(z >= v) >= top_k)
        keep = z >= kth
    if top_p < 1:
        e = np.exp((z - z.max()) / T) * keep
        S = e.sum()
        cands = [v for v in np.unique(z[keep]) if np.sum(e[z >= v]) / S >= top_p]
        keep &= z >= max(cands)
    return keep


@pytest.mark.parametrize("coarse", [False, True])
def test_brute_force_thresholds(coarse):
    rng = np.random.default_rng(3 + coarse)
    for trial in range(300):
        V = int(rng.integers(2, 12))
        z = rng.normal(0, 2, V)
        if coarse:                   # many ties, like bf16 logits
            z = np.round(z * 2) / 2
        T = float(rng.choice([0.5, 0.8, 1.0, 1.7]))
        top_k = int(rng.integers(0, V + 2))
        top_p = float(rng.choice([1.0, 0.3, 0.5, 0.9, 0.95, 0.99]))
        q, near = transformed_probs(z[None], T, top_k, top_p)
        if near[0]:
            continue
        keep = _brute_force_keep(z, T, top_k, top_p)
        np.testing.assert_array_equal(q[0] > 0, keep)
        e = np.exp((z - z.max()) / T) * keep
        np.testing.assert_allclose(q[0], e / e.sum(), rtol=1e-12)


def test_nucleus_near_tie_flag():
    # masses 0.5, 0.3, 0.2 -> mass of the top two is exactly 0.8
    z = np.log(np.array([[0.5, 0.3, 0.2]]))
    assert transformed_probs(z, 1.0, top_p=0.8)[1][0]
    assert transformed_probs(z, 1.0, top_p=0.8 + 1e-6)[1][0]
    assert not transformed_probs(z, 1.0, top_p=0.8 + 5e-6)[1][0]
    assert not transformed_probs(z, 1.0, top_p=0.79)[1][0]
