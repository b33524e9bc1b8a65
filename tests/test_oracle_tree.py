"""Pins of the oracle's REST tree verification.

"简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法" (REST),
section "REST: 基于检索的投机解码": drafts are paths of a trie laid out as a
BFS pseudo-sequence; a draft token is accepted iff it equals the token the
LLM would emit, so the result is exactly greedy decoding. Checked against
brute force over every root path and a sequential greedy walk.
"""

import numpy as np
import pytest

import oracle
import workloads


def _greedy_walk(z, tok, par):
    """Sequential greedy decoding through the tree: follow the child whose token
    is the argmax of the current node's row; stop when there is none."""
    N = tok.size
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[par[i]].append(i)
    node, path = 0, [0]
    while True:
        am = int(np.argmax(z[node]))
        nxt = [c for c in children[node] if tok[c] == am]
        if not nxt:
            return path, am
        node = nxt[0]
        path.append(node)


def _brute_force(z, tok, par):
    """Longest root path whose every token equals its parent's argmax."""
    N = tok.size
    best = (0, 0)
    for i in range(N):
        node, ok, d = i, True, 0
        while node > 0:
            if tok[node] != int(np.argmax(z[par[node]])):
                ok = False
            node = par[node]
            d += 1
        if ok and d > best[0]:
            best = (d, i)
    return best


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_matches_greedy_walk_and_brute_force(seed):
    B, N, V = 12, 40, 200
    z, tok, par, dep = workloads.tree_inputs(B, N, V, seed, force_p=0.9)
    r = oracle.verify_tree(z, tok, par, dep, max_depth=6)
    z, tok, par, dep = (t.numpy() for t in (z, tok, par, dep))
    assert (r["status"] == 0).all()
    for b in range(B):
        path, bonus = _greedy_walk(z[b], tok[b], par[b])
        assert r["accept_len"][b] == len(path) - 1
        assert list(r["path_nodes"][b, : len(path)]) == path
        assert r["bonus"][b] == bonus
        assert list(r["tokens"][b, : len(path)]) == [int(tok[b, n]) for n in path[1:]] + [bonus]
        d, _ = _brute_force(z[b], tok[b], par[b])
        assert d == r["accept_len"][b]


def test_hand_built_tree():
    # root -> (1: tok 5), (2: tok 7); 1 -> (3: tok 2); 2 -> (4: tok 9)
    V = 10
    par = np.array([[-1, 0, 0, 1, 2]])
    dep = np.array([[0, 1, 1, 2, 2]])
    tok = np.array([[0, 5, 7, 2, 9]])
    z = np.zeros((1, 5, V))
    z[0, 0, 7] = 1.0   # root predicts 7 -> node 2 accepted
    z[0, 2, 9] = 1.0   # node 2 predicts 9 -> node 4 accepted
    z[0, 4, 3] = 1.0   # node 4 predicts 3 -> bonus
    z[0, 1, 2] = 1.0   # node 1 would accept node 3, but node 1 is rejected
    r = oracle.verify_tree(z, tok, par, dep, max_depth=3)
    assert r["accept_len"][0] == 2
    assert list(r["path_nodes"][0]) == [0, 2, 4, -1]
    assert list(r["tokens"][0]) == [7, 9, 3, -1]
    assert r["bonus"][0] == 3
    # nothing accepted: the bonus is the root's argmax
    z[0, 0] = 0.0
    z[0, 0, 1] = 1.0
    r = oracle.verify_tree(z, tok, par, dep, max_depth=3)
    assert r["accept_len"][0] == 0 and list(r["tokens"][0]) == [1, -1, -1, -1]


def test_duplicate_siblings_lowest_index_wins():
    V = 6
    par = np.array([[-1, 0, 0, 1, 2]])
    dep = np.array([[0, 1, 1, 2, 2]])
    tok = np.array([[0, 4, 4, 1, 1]])
    z = np.zeros((1, 5, V))
    z[0, 0, 4] = 1
    z[0, 1, 1] = 1
    z[0, 2, 1] = 1
    r = oracle.verify_tree(z, tok, par, dep, max_depth=2)
    assert list(r["path_nodes"][0]) == [0, 1, 3]


def test_malformed_trees_are_rejected():
    V = 6
    z = np.zeros((5, 3, V))
    par = np.array([[-1, 0, 1], [0, 0, 1], [-1, 2, 1], [-1, 0, 0], [-1, 0, 1]])
    dep = np.array([[0, 1, 2], [0, 1, 2], [0, 1, 2], [0, 1, 2], [0, 1, 2]])
    tok = np.array([[0, 1, 2], [0, 1, 2], [0, 1, 2], [0, 1, 2], [0, 1, 7]])
    r = oracle.verify_tree(z, tok, par, dep, max_depth=2)
    # ok; parent[0] != -1; parent[1] >= 1; depth inconsistent; token out of range
    assert list(r["status"]) == [0, 4, 4, 4, 4]
    assert oracle.verify_tree(z[:1], tok[:1], par[:1], dep[:1], max_depth=1)["status"][0] == 4
