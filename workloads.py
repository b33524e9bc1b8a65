"""Seeded synthetic inputs for the verification workloads.

This module only draws random numbers and lays them out; it holds none of the
verification arithmetic. Both the CUDA path (tests, bench) and the CPU oracle
(tests) consume the tensors it makes, so the two sides always see the same
bytes. Logits are drawn with ``torch.Generator`` on the requested device (CPU
for the parity tests, the GPU for the large bench inputs); tree structure and
tokens use numpy's PCG64.

Workload recipes (shapes and distributions of the pages' experiments; the
pages' datasets and models are not available, these stand in for them):

* tiny         B=1, gamma=4, V=1000, f32, T=1. z_t ~ N(0, 2^2); z_d = z_t + N(0, 0.5^2).
* nucleus      B=8, gamma=4, V=32000, bf16, T=0.8, top_p=0.95.
               z_t ~ N(0, 3^2) plus 6 on a Bernoulli(0.01) token mask per row;
               z_d = z_t + N(0, sigma^2), sigma in {0.5, 1.5}; drawn in f32,
               rounded to bf16 (round-to-nearest-even).
* large_vocab  B=64, gamma=7, V=128256, f32, T in {0, 1}.
               z_t ~ N(0, 2.5^2) - 1.1 ln(rank_i), rank a seeded permutation
               of 1..V shared by all rows (a Zipf(1.1) log-frequency prior);
               z_d = z_t + N(0, 1).
* tree         B=16, N=64, V=32016, f32. A seeded random trie (depth <= 6,
               1-4 children per internal node, own counts ~ Poisson(5), node
               weight = count of its prefix = subtree sum), top-64 nodes by
               weight (ties: shallower, then creation order; ancestor-closed),
               laid out in BFS order. Sibling tokens distinct, uniform on V.
               z ~ N(0, 2^2); for each node with children, with probability
               0.7 one uniformly chosen child's token gets the row max + 1.
* mentor       B=32, gamma=5, V=32128, f32, T=1, D in {0.01, 0.1}.
               z_t ~ N(0, 2^2); z_d = z_t + N(0, 1.2^2).
* rest         the REST step: B=16 sequences, C=256 retrieved continuations
               of up to L=16 tokens each (a stand-in for datastore retrieval:
               12 base continuations per sequence, chosen with Zipf(1)
               popularity; each candidate copies its base up to a divergence
               point ~ Geometric(0.15) and continues with uniform tokens;
               lengths uniform in [L/2, L]); the draft tree of N=64 nodes is
               built from them and verified against [B, N, V=32016] f32
               logits z ~ N(0, 2^2), where, for each node with children,
               with probability 0.7 one uniformly chosen child's token gets
               the row max + 1.

Draft tokens for the parity tests are drawn by the oracle's sampler from the
transformed draft distribution. ``gumbel_drafts`` below is a stand-in draft
model for inputs too large for the oracle: it draws from softmax(z_d / T)
with the Gumbel-max construction (no top-k / top-p), so under a nucleus
transform a drafted token can fall outside the draft's nucleus.
"""

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(kind="linear", B=1, gamma=4, V=1000, dtype="f32", temperature=1.0,
                 top_p=1.0, top_k=0, steps=64, sd_t=2.0, sd_d=0.5),
    "nucleus": dict(kind="linear", B=8, gamma=4, V=32000, dtype="bf16", temperature=0.8,
                    top_p=0.95, top_k=0, steps=1000, sd_t=3.0, sd_d=0.5, boost=6.0,
                    boost_p=0.01),
    "large_vocab": dict(kind="linear", B=64, gamma=7, V=128256, dtype="f32", temperature=1.0,
                        top_p=1.0, top_k=0, steps=200, sd_t=2.5, sd_d=1.0, zipf=1.1),
    "tree": dict(kind="tree", B=16, N=64, V=32016, dtype="f32", sd=2.0, max_depth=6,
                 force_p=0.7),
    "mentor": dict(kind="mentor", B=32, gamma=5, V=32128, dtype="f32", temperature=1.0,
                   steps=500, sd_t=2.0, sd_d=1.2, kl_bound=0.1, iters=30),
    "rest": dict(kind="rest", B=16, N=64, V=32016, dtype="f32", C=256, L=16, bases=12,
                 diverge=0.15, sd=2.0, force_p=0.7),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def linear_logits(B, gamma, V, seed, dtype="f32", device="cpu", sd_t=2.0, sd_d=0.5,
                  boost=0.0, boost_p=0.0, zipf=0.0):
    """Target logits [B, gamma+1, V] and draft logits [B, gamma, V].

    Draft row k is target row k plus N(0, sd_d^2) noise. ``boost`` adds a
    constant on a Bernoulli(boost_p) mask; ``zipf`` subtracts s*ln(rank).
    """
    g = _gen(seed, device)
    zt = torch.randn(B, gamma + 1, V, generator=g, device=device, dtype=torch.float32) * sd_t
    if boost_p > 0:
        mask = torch.rand(B, gamma + 1, V, generator=g, device=device) < boost_p
        zt += boost * mask
    if zipf > 0:
        rank = torch.randperm(V, generator=g, device=device).to(torch.float32) + 1.0
        zt -= zipf * torch.log(rank)
    zd = zt[:, :gamma] + torch.randn(B, gamma, V, generator=g, device=device,
                                     dtype=torch.float32) * sd_d
    td = TORCH_DTYPE[dtype]
    return zt.to(td).contiguous(), zd.to(td).contiguous()


def config_logits(name, seed, steps=1, device="cpu", **over):
    """Logits for ``steps`` stacked steps of a named linear/mentor workload."""
    c = dict(CONFIGS[name])
    c.update(over)
    return linear_logits(c["B"] * steps, c["gamma"], c["V"], seed, dtype=c["dtype"],
                         device=device, sd_t=c["sd_t"], sd_d=c["sd_d"],
                         boost=c.get("boost", 0.0), boost_p=c.get("boost_p", 0.0),
                         zipf=c.get("zipf", 0.0))


def gumbel_drafts(draft, temperature, seed):
    """Stand-in draft model: x_k = argmax_i(z_d[k, i]/T + G_i), G ~ Gumbel(0, 1).

    Temperature 0 gives the plain argmax. Returns int32 [B, gamma] on the
    logits' device.
    """
    B, G, V = draft.shape
    if G == 0:
        return torch.zeros(B, 0, dtype=torch.int32, device=draft.device)
    if temperature == 0:
        return draft.float().argmax(dim=2).to(torch.int32)
    g = _gen(seed, draft.device)
    out = torch.empty(B, G, dtype=torch.int32, device=draft.device)
    chunk = max(1, (1 << 26) // (G * V))
    for s in range(0, B, chunk):
        z = draft[s:s + chunk].float() / temperature
        u = torch.rand(z.shape, generator=g, device=draft.device).clamp_(1e-12, 1.0)
        out[s:s + chunk] = (z - torch.log(-torch.log(u))).argmax(dim=2).to(torch.int32)
    return out


def _random_trie(rng, V, max_depth, n_min):
    """Random trie as lists (parent, depth, token, own_count) in creation order."""
    while True:
        parent, depth, token, count = [-1], [0], [int(rng.integers(V))], [0]
        frontier = [0]
        while frontier:
            nxt = []
            for node in frontier:
                if depth[node] >= max_depth:
                    continue
                if node != 0 and rng.random() < 0.25:
                    continue
                nch = int(rng.integers(1, 5))
                toks = rng.choice(V, size=nch, replace=False)
                for t in toks:
                    parent.append(node)
                    depth.append(depth[node] + 1)
                    token.append(int(t))
                    count.append(int(rng.poisson(5)))
                    nxt.append(len(parent) - 1)
            frontier = nxt
        if len(parent) >= n_min:
            return parent, depth, token, count


def tree_inputs(B, N, V, seed, max_depth=6, sd=2.0, force_p=0.7, device="cpu"):
    """BFS pseudo-sequences of top-N trie subtrees plus their target logits.

    Returns (target [B, N, V] f32, node_tokens, parent, depth) with the int
    arrays int32 [B, N]. Node 0 is the root; parent[0] = -1.
    """
    rng = np.random.default_rng(seed)
    toks = np.zeros((B, N), np.int32)
    par = np.zeros((B, N), np.int32)
    dep = np.zeros((B, N), np.int32)
    forced = []
    for b in range(B):
        parent, depth, token, count = _random_trie(rng, V, max_depth, N)
        M = len(parent)
        weight = np.array(count, dtype=np.int64)
        for i in range(M - 1, 0, -1):           # children are created after parents
            weight[parent[i]] += weight[i]
        order = sorted(range(M), key=lambda i: (-weight[i], depth[i], i))
        chosen = set(order[:N])
        children = [[] for _ in range(M)]
        for i in range(1, M):
            if i in chosen:
                children[parent[i]].append(i)
        bfs = [0]
        for node in bfs:
            bfs.extend(children[node])
        pos = {node: j for j, node in enumerate(bfs)}
        for j, node in enumerate(bfs):
            toks[b, j] = token[node]
            par[b, j] = -1 if node == 0 else pos[parent[node]]
            dep[b, j] = depth[node]
        for j, node in enumerate(bfs):
            ch = children[node]
            if ch and rng.random() < force_p:
                forced.append((b, j, token[ch[int(rng.integers(len(ch)))]]))
    g = _gen(seed, device)
    z = torch.randn(B, N, V, generator=g, device=device, dtype=torch.float32) * sd
    if forced:
        bi = torch.tensor([f[0] for f in forced], device=device)
        ji = torch.tensor([f[1] for f in forced], device=device)
        ti = torch.tensor([f[2] for f in forced], device=device)
        rowmax = z[bi, ji].max(dim=1).values
        z[bi, ji, ti] = rowmax + 1.0
    as_t = lambda a: torch.from_numpy(a).to(device)
    return z.contiguous(), as_t(toks), as_t(par), as_t(dep)


def rest_candidates(B, C, L, V, seed, bases=12, diverge=0.15):
    """Retrieved continuations [B, C, L] int32 (-1 after each one's end)."""
    rng = np.random.default_rng(seed)
    out = np.full((B, C, L), -1, np.int32)
    pop = 1.0 / np.arange(1, bases + 1)
    pop /= pop.sum()
    for b in range(B):
        base = rng.integers(0, V, (bases, L))
        pick = rng.choice(bases, size=C, p=pop)
        cut = np.minimum(rng.geometric(diverge, size=C), L)
        lens = rng.integers(L // 2, L + 1, size=C)
        fresh = rng.integers(0, V, (C, L))
        for c in range(C):
            row = np.where(np.arange(L) < cut[c], base[pick[c]], fresh[c])
            out[b, c, :lens[c]] = row[:lens[c]]
    return out


def forced_tree_logits(node_tokens, parent, n_nodes, V, seed, sd=2.0, force_p=0.7, device="cpu"):
    """Logits [B, N, V] f32 ~ N(0, sd^2) for a built tree; for each node with
    children, with probability force_p one uniformly chosen child's token gets
    the row max + 1 (so the greedy walk descends)."""
    tok = np.asarray(node_tokens)
    par = np.asarray(parent)
    B, N = tok.shape
    rng = np.random.default_rng(seed)
    forced = []
    for b in range(B):
        kids = [[] for _ in range(N)]
        for i in range(1, int(n_nodes[b])):
            kids[par[b, i]].append(i)
        for j in range(N):
            if kids[j] and rng.random() < force_p:
                forced.append((b, j, int(tok[b, kids[j][int(rng.integers(len(kids[j])))]])))
    g = _gen(seed, device)
    z = torch.randn(B, N, V, generator=g, device=device, dtype=torch.float32) * sd
    if forced:
        bi = torch.tensor([f[0] for f in forced], device=device)
        ji = torch.tensor([f[1] for f in forced], device=device)
        ti = torch.tensor([f[2] for f in forced], device=device)
        z[bi, ji, ti] = z[bi, ji].max(dim=1).values + 1.0
    return z.contiguous()


def algorithmic_bytes(kind, B, V, esize, gamma=0, N=0, temperature=1.0):
    """Bytes of logits one verification step must read (each row once).

    T > 0: all 2*gamma+1 rows; T = 0: the gamma+1 target rows; trees: N rows.
    """
    if kind in ("tree", "rest"):
        rows = N
    elif temperature == 0:
        rows = gamma + 1
    else:
        rows = 2 * gamma + 1
    return B * rows * V * esize


def verified_positions(kind, B, gamma=0, N=0):
    """Positions a step verifies: B*gamma (linear), B*(N-1) (tree, rest)."""
    return B * (N - 1) if kind in ("tree", "rest") else B * gamma


def l2_flush_bytes():
    """A buffer size comfortably larger than a GB300 L2 (129 MB)."""
    return 512 * 1024 * 1024


__all__ = ["CONFIGS", "linear_logits", "config_logits", "gumbel_drafts", "tree_inputs", "rest_candidates",
           "forced_tree_logits",
           "algorithmic_bytes", "verified_positions", "l2_flush_bytes"]
