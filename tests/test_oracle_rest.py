"""Pins for the oracle's REST draft-tree construction.

[REST] "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法", section
"REST: 基于检索的投机解码": trie nodes are the candidates' prefixes weighted by
how often they occur, the draft tree is the subtree of the heaviest nodes, its
breadth-first walk is the pseudo-sequence, and the attention mask restores
each token's ancestry. Pinned by the page's own example (hand-counted), by a
brute force that enumerates every token tuple instead of walking candidates,
and by the structural invariants the page states (every draft sequence is a
root path of the tree; parents precede children in the pseudo-sequence).
"""

import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rest_trie_example.txt")


def _golden():
    g = {"N": {}}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "V":
            g["V"] = int(rest)
        elif key == "root":
            g["root"] = int(rest)
        elif key == "candidates":
            g["cands"] = [[int(t) for t in c.split()] for c in rest.split(";")]
        elif key == "weights":
            g["weights"] = {tuple(int(t) for t in k.split(",")): int(v)
                            for k, v in (w.split(":") for w in rest.split())}
        elif key.startswith("N="):
            parts = [p.split() for p in rest.split("|")]
            g["N"][int(key[2:])] = [list(map(int, p)) for p in parts]
    return g


def _pad(cands, L):
    return np.array([c + [-1] * (L - len(c)) for c in cands], np.int64)


def test_page_example():
    g = _golden()
    cands = _pad(g["cands"], 4)
    # the hand count of the fixture: every prefix with its occurrences
    for path, w in g["weights"].items():
        assert sum(tuple(c[:len(path)]) == path for c in g["cands"]) == w
    assert len(g["weights"]) == len({tuple(c[:l]) for c in g["cands"] for l in range(1, len(c) + 1)})
    for N, (toks, par, dep, (n,)) in g["N"].items():
        r = oracle.rest_tree(cands, None, g["root"], N, g["V"])
        assert r["status"] == 0
        np.testing.assert_array_equal(r["tokens"], toks)
        np.testing.assert_array_equal(r["parent"], par)
        np.testing.assert_array_equal(r["depth"], dep)
        assert r["n_nodes"] == n


def _brute(cands, counts, N, V):
    """Every token tuple up to length L, weights by direct comparison."""
    C, L = cands.shape
    seqs = []
    for c in range(C):
        row = list(cands[c])
        end = row.index(-1) if -1 in row else L
        seqs.append((tuple(row[:end]), counts[c]))
    nodes = {}
    for l in range(1, L + 1):
        for path in itertools.product(range(V), repeat=l):
            hits = [m for s, m in seqs if len(s) >= l and s[:l] == path]
            if hits:
                nodes[path] = sum(hits)
    return nodes


@pytest.mark.parametrize("seed", range(12))
def test_brute_force_weights_and_choice(seed):
    rng = np.random.default_rng(seed)
    C, L, V = int(rng.integers(1, 7)), int(rng.integers(1, 5)), int(rng.integers(2, 4))
    cands = rng.integers(0, V, (C, L))
    for c in range(C):                        # ragged ends
        e = int(rng.integers(0, L + 1))
        cands[c, e:] = -1
    counts = rng.integers(0, 4, C)
    nodes = _brute(cands, counts, 0, V)
    for N in (2, 3, 5, 9, 40):
        r = oracle.rest_tree(cands, counts, 1, N, V)
        n = r["n_nodes"]
        assert n == 1 + min(N - 1, len(nodes))
        paths = []
        for i in range(1, n):
            path, j = [], i
            while j > 0:
                path.append(int(r["tokens"][j]))
                j = r["parent"][j]
            paths.append(tuple(reversed(path)))
        # exactly the top N-1 nodes of the stated ranking
        key = lambda t: (-nodes[t], len(t), t)
        want = sorted(nodes, key=key)[:N - 1]
        assert sorted(paths, key=key) == want
        # positions follow (length, path)
        assert paths == sorted(paths, key=lambda t: (len(t), t))
        for i, t in enumerate(paths):
            assert r["depth"][i + 1] == len(t)


@pytest.mark.parametrize("seed", range(8))
def test_structure_and_mask(seed):
    rng = np.random.default_rng(100 + seed)
    C, L, V, N = 24, 6, 5, 32
    cands = rng.integers(0, V, (C, L))
    cands[:, int(rng.integers(2, L)):][rng.random(C) < 0.4] = -1
    r = oracle.rest_tree(cands, None, 3, N, V)
    n = r["n_nodes"]
    par, dep, tok = r["parent"], r["depth"], r["tokens"]
    assert par[0] == -1 and dep[0] == 0 and tok[0] == 3
    for i in range(1, n):
        assert 0 <= par[i] < i and dep[i] == dep[par[i]] + 1
        assert dep[i] >= dep[i - 1]
    # siblings in ascending token order, distinct (a trie)
    for a in range(n):
        kids = [tok[i] for i in range(1, n) if par[i] == a]
        assert kids == sorted(kids) and len(set(kids)) == len(kids)
    # mask = ancestor-or-self, from walking the parents
    want = np.zeros((N, N), np.uint8)
    for i in range(n):
        j = i
        while j >= 0:
            want[i, j] = 1
            j = par[j]
    np.testing.assert_array_equal(r["mask"], want)
    assert (tok[n:] == -1).all() and (par[n:] == -1).all() and (dep[n:] == -1).all()
    # every candidate's prefix, down to the deepest chosen one, is a root path
    path_of = {}
    for i in range(n):
        path, j = [], i
        while j > 0:
            path.append(int(tok[j]))
            j = par[j]
        path_of[tuple(reversed(path))] = i
    for c in range(C):
        row = list(cands[c])
        end = row.index(-1) if -1 in row else L
        l = 0
        while l < end and tuple(row[:l + 1]) in path_of:
            l += 1
        assert all(tuple(row[:k]) in path_of for k in range(l + 1))


def test_data_errors_and_degenerate_inputs():
    V = 10
    ok = np.array([[1, 2, -1], [1, 3, 4]])
    assert oracle.rest_tree(ok, None, 0, 4, V)["status"] == 0
    for bad in (np.array([[1, 10, -1]]), np.array([[1, -2, -1]])):
        r = oracle.rest_tree(bad, None, 0, 4, V)
        assert r["status"] == 4 and r["n_nodes"] == -1 and (r["tokens"] == -1).all() and not r["mask"].any()
    assert oracle.rest_tree(ok, None, V, 4, V)["status"] == 4                 # root out of range
    assert oracle.rest_tree(ok, np.array([1, -1]), 0, 4, V)["status"] == 4   # negative count
    assert oracle.rest_tree(ok, np.array([1, oracle.REST_MAX_COUNT]), 0, 4, V)["status"] == 4
    # every candidate empty: the root alone
    r = oracle.rest_tree(np.full((3, 4), -1), None, 5, 4, V)
    assert r["n_nodes"] == 1 and list(r["tokens"]) == [5, -1, -1, -1] and r["mask"][0, 0] == 1
    # tokens after a candidate's end are ignored
    a = oracle.rest_tree(np.array([[1, -1, 7]]), None, 0, 4, V)
    assert a["n_nodes"] == 2 and a["tokens"][1] == 1
    # zero multiplicity keeps the node (it occurs) with weight 0: ranked last
    r = oracle.rest_tree(np.array([[1, -1], [2, -1]]), np.array([0, 1]), 0, 2, V)
    assert r["n_nodes"] == 2 and r["tokens"][1] == 2
    # identical candidates add up
    r = oracle.rest_tree(np.array([[4, -1], [4, -1], [3, -1]]), None, 0, 2, V)
    assert r["tokens"][1] == 4
