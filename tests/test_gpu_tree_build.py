"""REST draft-tree construction on the GPU (spec_tree_build) against the
oracle, element by element (integer work: bit-exact), then the built trees
through spec_verify_tree against the oracle's verify_tree.

[REST] "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法", section
"REST: 基于检索的投机解码".
"""

import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_05_gb300 as sv
import workloads

pytestmark = pytest.mark.gpu

KEYS = ("node_tokens", "parent", "depth", "n_nodes", "status")
ORACLE_KEY = {"node_tokens": "tokens", "parent": "parent", "depth": "depth", "n_nodes": "n_nodes",
              "status": "status"}


def _compare(cand, counts, root, N, V, with_mask=True, label=""):
    g = sv.tree_build(torch.from_numpy(cand).cuda(), torch.from_numpy(root).cuda(), V, N,
                      counts=None if counts is None else torch.from_numpy(counts).cuda(),
                      with_mask=with_mask)
    r = oracle.rest_tree_batch(cand, counts, root, N, V)
    for k in KEYS:
        np.testing.assert_array_equal(g[k].cpu().numpy(), r[ORACLE_KEY[k]], err_msg=f"{label} {k}")
    if with_mask:
        np.testing.assert_array_equal(g["mask"].cpu().numpy(), r["mask"], err_msg=f"{label} mask")
    return g, r


def _random_case(rng, B, C, L, V, ragged=True):
    cand = rng.integers(0, V, (B, C, L)).astype(np.int32)
    if ragged:
        ends = rng.integers(0, L + 1, (B, C))
        cand[np.arange(L)[None, None, :] >= ends[:, :, None]] = -1
    return cand


@pytest.mark.parametrize("seed", range(6))
def test_small_random_trees(seed):
    rng = np.random.default_rng(seed)
    B, C, L, V = 7, int(rng.integers(1, 60)), int(rng.integers(1, 10)), int(rng.integers(2, 7))
    cand = _random_case(rng, B, C, L, V)
    counts = rng.integers(0, 5, (B, C)).astype(np.int32)
    root = rng.integers(0, V, B).astype(np.int32)
    for N in (2, 5, 17, 64, 200):
        _compare(cand, counts, root, N, V, label=f"seed {seed} N {N}")
        _compare(cand, None, root, N, V, label=f"seed {seed} N {N} unit counts")


def test_page_example_on_gpu():
    cand = np.array([[[11, 12, -1, -1], [11, 12, 13, -1], [11, 14, -1, -1]]], np.int32)
    g, _ = _compare(cand, None, np.array([7], np.int32), 5, 100)
    assert list(g["node_tokens"][0].cpu().numpy()) == [7, 11, 12, 14, 13]
    assert list(g["parent"][0].cpu().numpy()) == [-1, 0, 1, 1, 2]


@pytest.mark.parametrize("C,L,N", [(1024, 4, 1024), (128, 32, 1024), (4096 // 32, 32, 97), (1, 1, 2),
                                   (1024, 1, 1024), (1, 32, 1024)])
def test_limits(C, L, N):
    rng = np.random.default_rng(C * 31 + L)
    V = 3 if C > 1 else 1000
    cand = _random_case(rng, 3, C, L, V, ragged=L > 1)
    counts = rng.integers(0, 1 << 20, (3, C)).astype(np.int32)
    root = np.array([0, 1, 2], np.int32)
    _compare(cand, counts, root, N, V, label=f"C {C} L {L} N {N}")


def test_mask_layouts_and_degenerate_inputs():
    rng = np.random.default_rng(5)
    V = 6
    cand = _random_case(rng, 4, 20, 5, V)
    root = np.array([1, 2, 3, 4], np.int32)
    for N in (5, 6, 7, 33):                  # N % 4 != 0: byte stores
        _compare(cand, None, root, N, V, label=f"N {N}")
    _compare(cand, None, root, 8, V, with_mask=False, label="no mask")
    # empty candidates, identical candidates, zero multiplicities
    deg = np.full((3, 6, 4), -1, np.int32)
    deg[1, :, :2] = [3, 4]
    deg[2, :3, :3] = [[1, 2, 3], [1, 2, 5], [2, 2, 2]]
    counts = np.array([[1] * 6, [0] * 6, [0, 2, 1, 0, 0, 0]], np.int32)
    g, _ = _compare(deg, counts, np.array([0, 0, 0], np.int32), 6, V, label="degenerate")
    assert list(g["n_nodes"].cpu().numpy()) == [1, 3, 6]


def test_data_errors_are_per_sequence():
    V = 10
    cand = np.tile(np.array([[1, 2, -1], [1, 3, 4]], np.int32), (5, 1, 1))
    cand[1, 0, 1] = V            # token out of range
    cand[2, 1, 2] = -2           # below -1
    root = np.array([0, 0, 0, V, 0], np.int32)   # sequence 3: root out of range
    counts = np.ones((5, 2), np.int32)
    counts[4, 1] = -1            # sequence 4: negative multiplicity
    g, _ = _compare(cand, counts, root, 6, V, label="errors")
    assert list(g["status"].cpu().numpy()) == [0, 4, 4, 4, 4]


def test_host_buffers_end_to_end():
    rng = np.random.default_rng(9)
    cand = _random_case(rng, 2, 30, 6, 4)
    g = sv.tree_build(torch.from_numpy(cand), torch.tensor([1, 2], dtype=torch.int32), 4, 16)
    r = oracle.rest_tree_batch(cand, None, np.array([1, 2]), 16, 4)
    assert g["node_tokens"].device.type == "cpu"
    np.testing.assert_array_equal(g["node_tokens"].numpy(), r["tokens"])
    np.testing.assert_array_equal(g["mask"].numpy(), r["mask"])


def test_rest_step_build_then_verify():
    """The REST step at the workload's sizes: trees built on the GPU from the
    synthetic retrieval, checked against the oracle, then verified greedily
    against logits whose forced children make the walk descend."""
    c = workloads.CONFIGS["rest"]
    B, N, V, C, L = c["B"], c["N"], c["V"], c["C"], c["L"]
    cand = workloads.rest_candidates(B, C, L, V, seed=11, bases=c["bases"], diverge=c["diverge"])
    root = np.arange(B, dtype=np.int32)
    g, r = _compare(cand, None, root, N, V, label="rest workload")
    assert (r["n_nodes"] == N).all()
    z = workloads.forced_tree_logits(r["tokens"], r["parent"], r["n_nodes"], V, seed=11, device="cuda")
    out = sv.verify_tree(z, g["node_tokens"], g["parent"], g["depth"], L)
    ref = oracle.verify_tree(z.cpu().numpy(), r["tokens"], r["parent"], r["depth"], L)
    np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
    np.testing.assert_array_equal(out["tokens"].cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(out["path_nodes"].cpu().numpy(), ref["path_nodes"])
    assert ref["accept_len"].mean() > 1.0
