"""REST draft-tree construction (test infrastructure; see the package header).

[REST] "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法", section
"REST: 基于检索的投机解码": the continuations retrieved for the context are
the candidate sequences; every prefix of a candidate is a node of a trie whose
weight is the number of times that prefix occurs among the candidates; the
most frequent prefixes come from the subtree of the heaviest nodes; a
breadth-first walk of that subtree gives the pseudo-sequence the target model
scores, and an attention mask restores each token's own ancestry (tree
attention).

Readings where the page is silent (each also listed in the design notes):

* A candidate ends at its first -1; every entry must be -1 or a token in
  [0, V), every multiplicity in [0, 2^20), the root token in [0, V);
  otherwise the sequence is a data error.
* Weight of a prefix = the sum of the multiplicities of the candidates that
  start with it (multiplicity 1 when none are given).
* The subtree: the N - 1 prefixes ranked first by (weight descending, length
  ascending, token path lexicographically ascending). A prefix never
  outweighs its own prefixes and is longer, so the chosen set is closed
  under taking parents.
* Breadth-first order: the root (the context's last token) at position 0,
  then the chosen prefixes by (length, path) -- the BFS that visits each
  node's children in ascending token order.
* mask[i][j] = 1 iff node j is node i or one of its ancestors.
* Fewer than N - 1 distinct prefixes: n_nodes = 1 + their number; the
  remaining positions hold token, parent and depth -1 and an all-zero mask
  row.

Plain Python over tuples: no trie structure beyond a dictionary of prefixes.
"""

import numpy as np

MAX_COUNT = 1 << 20


def _sequence(candidates, counts, root_token, V):
    """(list of (tokens tuple, multiplicity), ok) for one sequence."""
    cands = np.asarray(candidates).astype(np.int64)
    C = cands.shape[0]
    mult = np.ones(C, np.int64) if counts is None else np.asarray(counts).astype(np.int64)
    ok = 0 <= int(root_token) < V
    ok = ok and bool(np.all((cands >= -1) & (cands < V)))
    ok = ok and bool(np.all((mult >= 0) & (mult < MAX_COUNT)))
    seqs = []
    for c in range(C):
        row = [int(t) for t in cands[c]]
        end = row.index(-1) if -1 in row else len(row)
        seqs.append((tuple(row[:end]), int(mult[c])))
    return seqs, ok


def rest_tree(candidates, counts, root_token, N, V):
    """One sequence: candidates [C, L] int, counts [C] or None.

    Returns dict(tokens [N], parent [N], depth [N] int32, mask [N, N] uint8,
    n_nodes, status) with status 0 (ok) or 4 (data error; every output -1 and
    the mask zero).
    """
    tokens = np.full(N, -1, np.int32)
    parent = np.full(N, -1, np.int32)
    depth = np.full(N, -1, np.int32)
    mask = np.zeros((N, N), np.uint8)
    seqs, ok = _sequence(candidates, counts, root_token, V)
    if not ok:
        return dict(tokens=tokens, parent=parent, depth=depth, mask=mask, n_nodes=-1, status=4)
    # weight of every prefix (a trie node)
    weight = {}
    for toks, m in seqs:
        for l in range(1, len(toks) + 1):
            weight[toks[:l]] = weight.get(toks[:l], 0) + m
    ranked = sorted(weight, key=lambda path: (-weight[path], len(path), path))
    chosen = ranked[:N - 1]
    order = sorted(chosen, key=lambda path: (len(path), path))
    pos = {(): 0}
    for i, path in enumerate(order):
        pos[path] = i + 1
    tokens[0] = int(root_token)
    depth[0] = 0
    for path, i in pos.items():
        if not path:
            continue
        tokens[i] = path[-1]
        depth[i] = len(path)
        parent[i] = pos[path[:-1]]
    for path, i in pos.items():
        for l in range(len(path) + 1):
            mask[i, pos[path[:l]]] = 1
    return dict(tokens=tokens, parent=parent, depth=depth, mask=mask, n_nodes=len(pos), status=0)


def rest_tree_batch(candidates, counts, root_token, N, V):
    """Batched rest_tree: candidates [B, C, L], counts [B, C] or None, root [B]."""
    cands = np.asarray(candidates)
    B = cands.shape[0]
    outs = [rest_tree(cands[b], None if counts is None else np.asarray(counts)[b],
                      int(np.asarray(root_token)[b]), N, V) for b in range(B)]
    return dict(tokens=np.stack([o["tokens"] for o in outs]),
                parent=np.stack([o["parent"] for o in outs]),
                depth=np.stack([o["depth"] for o in outs]),
                mask=np.stack([o["mask"] for o in outs]),
                n_nodes=np.array([o["n_nodes"] for o in outs], np.int32),
                status=np.array([o["status"] for o in outs], np.int32))
