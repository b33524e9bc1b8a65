"""fp64 restatement of the verification step and its two variants.

TEST INFRASTRUCTURE (see the package docstring): a plain, slow CPU oracle.
Every function cites the passage it follows. Vectorised over the batch with
numpy; loops run over draft positions, tree nodes and mentor rows only.

Readings taken where the pages are silent:

* q is the target distribution, p the draft one ([SpS], [Mentor]); the
  [SD] write-up swaps the letters and is rewritten into this notation.
* Sampling transforms ([SpS] "与标准采样方法的兼容性": apply nucleus,
  top-k and temperature before the scheme; [SD] "标准化采样框架") act on
  both q and p, in the order temperature -> top-k -> top-p. Selection uses
  raw logit values (monotone in z/T for T > 0). top-k keeps every value at
  least the k-th largest (tie-inclusive). top-p keeps the values z >= tau,
  where tau is the largest logit value whose cumulative mass (of the top-k
  renormalised distribution) reaches top_p; the crossing value and all of
  its ties are kept. top_k = 0 or top_k >= V and top_p >= 1 mean "off".
* Temperature 0 is argmax (lowest index on ties), the [SD] "argmax"
  sampling mode.
* Acceptance compares u < min(1, q(x)/p(x)); p(x) = 0 gives rho = +inf
  when q(x) > 0 and rho = 0 when q(x) = 0.
* Resampling and the bonus token use the inverse CDF in index order: the
  smallest i with C_i > u' * W. If rounding leaves no such i, the largest i
  with w_i > 0. A rejection with W = sum (q-p)+ = 0 (probability zero in
  exact arithmetic) samples from q instead.
* Rows holding NaN or +inf, or only -inf, are input errors (status 4);
  -inf alone is an ordinary zero-probability logit.
"""

import numpy as np

from .philox import uniform, PURPOSE_ACCEPT, PURPOSE_RESAMPLE, PURPOSE_DRAFT

NEAR_TIE = 1e-5
# Band of the top-p threshold decision (relative to the kept mass): the GPU's
# cumulative masses at the crossing are fp32 sums of the few head bins above it,
# accurate to a few 1e-7; a 1e-5 band would flag most rows of a large flat
# nucleus, where single tokens carry ~1e-5 of the mass.
THRESH_NEAR = 2e-6
STATUS_OK = 0
STATUS_EDATA = 4


def _f64(a):
    """Exact fp64 copy of a float32/bf16/float64 array or CPU/GPU tensor."""
    if hasattr(a, "detach"):
        return a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def _bad_rows(z):
    """[..., V] -> [...] True where a row holds NaN or +inf, or only -inf."""
    return np.isnan(z).any(-1) | np.isposinf(z).any(-1) | np.isneginf(z).all(-1)


# ---------------------------------------------------------------------------
# Sampling transforms: [SpS] "与标准采样方法的兼容性"; [SD] "标准化采样框架".
# ---------------------------------------------------------------------------

def transformed_probs(z, temperature, top_k=0, top_p=1.0):
    """Per-row probabilities after temperature, top-k and top-p.

    z: [R, V] logits. Returns (probs [R, V] fp64, near_tie [R] bool). The
    near-tie flag marks rows whose top-p threshold is decided by a cumulative
    mass within THRESH_NEAR of top_p (at the kept crossing value or at the
    next larger value), where fp32 and fp64 may legitimately choose
    differently.
    """
    z = _f64(z)
    R, V = z.shape
    near = np.zeros(R, dtype=bool)
    if temperature == 0:
        q = np.zeros_like(z)
        q[np.arange(R), np.argmax(z, axis=1)] = 1.0
        return q, near
    with np.errstate(invalid="ignore", over="ignore"):
        keep = np.ones_like(z, dtype=bool)
        if 0 < top_k < V:
            kth = -np.sort(-z, axis=1)[:, top_k - 1]
            keep = z >= kth[:, None]
        m = z.max(axis=1, keepdims=True)
        e = np.exp((z - m) / temperature) * keep
        if top_p < 1.0:
            s_k = e.sum(axis=1)
            order = np.argsort(-z, axis=1, kind="stable")
            zs = np.take_along_axis(z, order, axis=1)
            cs = np.cumsum(np.take_along_axis(e, order, axis=1), axis=1)
            frac = cs / s_k[:, None]
            last = np.ones_like(zs, dtype=bool)           # last element of a tie group
            last[:, :-1] = zs[:, 1:] != zs[:, :-1]
            ok = last & (frac >= top_p)
            j = np.where(ok.any(axis=1), np.argmax(ok, axis=1), V - 1)
            rows = np.arange(R)
            tau = zs[rows, j]
            idx = np.where(last, np.arange(V)[None, :], -1)
            prev_last = np.full((R, V), -1)
            prev_last[:, 1:] = np.maximum.accumulate(idx, axis=1)[:, :-1]
            jp = prev_last[rows, j]
            near = (frac[rows, j] - top_p) <= THRESH_NEAR
            near |= (jp >= 0) & ((top_p - frac[rows, np.maximum(jp, 0)]) <= THRESH_NEAR)
            keep &= z >= tau[:, None]
            e = e * keep
        q = e / e.sum(axis=1, keepdims=True)
    return q, near


# ---------------------------------------------------------------------------
# Modified rejection sampling: [SpS] "改进的拒绝采样".
# ---------------------------------------------------------------------------

def accept_test(u, q_x, p_x):
    """Accept draft token x with probability min(1, q(x)/p(x)).

    [SpS] "改进的拒绝采样", acceptance-probability equation; [SD]
    "接受-拒绝规则". Returns (accept, rho, near_tie) with near_tie when
    |u - min(1, rho)| <= NEAR_TIE.
    """
    u, q_x, p_x = (np.asarray(v, dtype=np.float64) for v in (u, q_x, p_x))
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = np.where(p_x > 0, q_x / np.where(p_x > 0, p_x, 1.0), np.where(q_x > 0, np.inf, 0.0))
    thr = np.minimum(1.0, rho)
    return u < thr, rho, np.abs(u - thr) <= NEAR_TIE


def inverse_cdf(u, w):
    """Index sampled from weights w [R, V] >= 0 with uniform u [R].

    The smallest i with C_i > u * W (C the inclusive prefix sum in index
    order, W = C_{V-1}); if rounding leaves none, the largest i with w_i > 0.
    This is the draw x ~ (f)_+ of [SpS] "改进的拒绝采样" once the weights are
    max(0, q - p), and the ordinary draw from q for the bonus token.
    Returns (index [R], near_tie [R]) with near_tie when u*W lies within
    NEAR_TIE * W of the boundary that decided the index (``admissible_draws``
    lists every index such a draw may return).
    """
    w = np.asarray(w, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    R, V = w.shape
    C = np.cumsum(w, axis=1)
    W = C[:, -1]
    t = u * W
    gt = C > t[:, None]
    rows = np.arange(R)
    has = gt.any(axis=1)
    pos = w > 0
    last_pos = V - 1 - np.argmax(pos[:, ::-1], axis=1)
    i = np.where(has, np.argmax(gt, axis=1), last_pos)
    lower = np.where(i > 0, C[rows, np.maximum(i - 1, 0)], -np.inf)
    near_hi = (C[rows, i] - t) <= NEAR_TIE * W
    near_lo = (t - lower) <= NEAR_TIE * W
    return i, near_hi | near_lo | ~has


ADM_K = 16


def admissible_draws(u, w, k=ADM_K):
    """Every index an inverse-CDF draw (``inverse_cdf``) from weights w [R, V]
    returns when its threshold t = u W moves by at most b = NEAR_TIE * W: the
    positive-weight indices j with C_{j-1} <= t + b and C_j > t - b (C the
    inclusive prefix sum, C_{-1} = 0), and the last positive-weight index
    when t + b reaches W (the rounding fallback). A draw computed in lower
    precision, whose prefix sums are within the band, returns one of them.

    Returns (adm [R, k] ascending, -1 padded; over [R] True where more than k
    indices qualify, which leaves the draw undecided by this check).
    """
    w = np.asarray(w, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    R, V = w.shape
    C = np.cumsum(w, axis=1)
    W = C[:, -1]
    t = u * W
    b = NEAR_TIE * W
    Cm = np.concatenate([np.zeros((R, 1)), C[:, :-1]], axis=1)
    pos = w > 0
    ok = pos & (Cm <= (t + b)[:, None]) & (C > (t - b)[:, None])
    last_pos = V - 1 - np.argmax(pos[:, ::-1], axis=1)
    rows = np.arange(R)
    fall = (t + b >= W) & pos.any(axis=1)
    ok[rows[fall], last_pos[fall]] = True
    cnt = ok.sum(axis=1)
    first = np.argsort(~ok, axis=1, kind="stable")[:, :k]   # the qualifying indices, ascending
    adm = np.where(np.take_along_axis(ok, first, axis=1), first, -1).astype(np.int64)
    if adm.shape[1] < k:
        adm = np.concatenate([adm, np.full((R, k - adm.shape[1]), -1, dtype=np.int64)], axis=1)
    return adm, cnt > k


def _merge_adm(a, b, k=ADM_K):
    """Union of two admissible sets [R, k] (ascending, -1 padded); over where
    the union exceeds k."""
    out = np.full_like(a, -1)
    over = np.zeros(a.shape[0], dtype=bool)
    for r in range(a.shape[0]):
        u = np.union1d(a[r][a[r] >= 0], b[r][b[r] >= 0])
        over[r] = u.size > k
        out[r, :min(k, u.size)] = u[:k]
    return out, over


def _emit(x, n, token):
    """tokens[b] = x[b, :n_b] followed by the resampled/bonus token, -1 padded."""
    B, gamma = x.shape
    pos = np.arange(gamma + 1)[None, :]
    xp = np.concatenate([x, np.full((B, 1), -1, dtype=np.int64)], axis=1)
    tokens = np.where(pos < n[:, None], xp, -1)
    tokens[np.arange(B), n] = token
    return tokens


def _uniform_fn(seed, uniform_fn):
    if uniform_fn is not None:
        return uniform_fn
    return lambda rows, pos, purpose: uniform(seed, rows, pos, purpose)


def verify(target, draft, draft_tokens, temperature=1.0, top_p=1.0, top_k=0,
           seed=0, offset=0, uniform_fn=None, lenience=1.0):
    """Batched speculative verification (modified rejection sampling).

    target [B, gamma+1, V], draft [B, gamma, V] (unused when temperature is
    0), draft_tokens [B, gamma]. Follows [SpS] "改进的拒绝采样": left to right,
    accept x_k with probability min(1, q_k(x_k)/p_k(x_k)); at the first
    rejection n resample from (q_n - p_n)_+ and stop; if all gamma are
    accepted, draw the bonus token from q_gamma (second bullet of that
    section; [SD] "至多 gamma+1 个 token").

    Temperature 0: q_k and p_k are one-hot at their argmaxes, so rho is 1
    when x_k is the target argmax and 0 otherwise (p(x)=0 when the draft
    token is not the draft argmax gives +inf or 0 by the same test), and the
    residual (q-p)_+ is one-hot at the target argmax (or zero, which falls
    back to q, the same token). Hence: accept iff x_k = argmax(target_k) and
    emit argmax(target_n); draft logits are not read.

    Uniforms: u_k = U(seed, offset+b, k, ACCEPT), u'_n = U(seed, offset+b,
    n, RESAMPLE); ``uniform_fn(rows, pos, purpose)`` may replace them.

    ``lenience`` l in ]0, 1] is the lenient variant of [SD] "方法细节"
    (extension in its appendix F): the draft probability is scaled by l
    before the comparison, so x_k is accepted with probability
    min(1, q(x)/(l p(x))), and a rejection resamples from
    norm(max(0, q - l p)). No token is then emitted with probability above
    q(x)/l (the guarantee that section states); l = 1 is the exact method.
    The pages state only the scaled comparison and the bound; the residual
    max(0, q - l p) is the reading that keeps the bound and reduces to
    (q - p)+ at l = 1. Temperature 0 is unaffected (one-hot rows give the
    same decisions for every l).

    Returns a dict: accepted [B], tokens [B, gamma+1] (-1 padded),
    next_token [B], status [B], near_tie [B] (a decision within the near-tie
    band: the row is excluded from exact comparison), adm_tokens [B, ADM_K]
    (every token the final draw may return when its threshold moves within
    the near-tie band, ``admissible_draws``; next_token is one of them),
    q_x / p_x [B, gamma] (the probabilities of each draft token), prob_near
    [B, gamma] (top-p threshold near-tie in either row at that position).
    """
    zt = _f64(target)
    B, G1, V = zt.shape
    gamma = G1 - 1
    x = np.asarray(draft_tokens, dtype=np.int64).reshape(B, gamma)
    U = _uniform_fn(seed, uniform_fn)
    rows = np.uint64(offset) + np.arange(B, dtype=np.uint64)

    bad = _bad_rows(zt).any(axis=1) | ((x < 0) | (x >= V)).any(axis=1)
    zd = None
    if temperature != 0:
        zd = _f64(draft).reshape(B, gamma, V)
        if gamma:
            bad |= _bad_rows(zd).any(axis=1)
    xs = np.clip(x, 0, V - 1)

    n = np.full(B, gamma, dtype=np.int64)
    token = np.full(B, -1, dtype=np.int64)
    adm = np.full((B, ADM_K), -1, dtype=np.int64)
    near = np.zeros(B, dtype=bool)
    q_x = np.full((B, gamma), np.nan)
    p_x = np.full((B, gamma), np.nan)
    prob_near = np.zeros((B, gamma), dtype=bool)
    brange = np.arange(B)

    if temperature == 0:
        am = np.argmax(zt, axis=2)
        match = xs == am[:, :gamma]
        q_x[:] = match
        p_x[:] = 1.0
        n = np.where(match.all(axis=1), gamma, np.argmin(match, axis=1)) if gamma else n
        token = am[brange, n]
        adm[:, 0] = token
    else:
        for k in range(gamma):
            q, nq = transformed_probs(zt[:, k], temperature, top_k, top_p)
            p, npd = transformed_probs(zd[:, k], temperature, top_k, top_p)
            q_x[:, k] = q[brange, xs[:, k]]
            p_x[:, k] = p[brange, xs[:, k]]
            prob_near[:, k] = nq | npd
            acc, _, near_acc = accept_test(U(rows, k, PURPOSE_ACCEPT), q_x[:, k], lenience * p_x[:, k])
            live = n == gamma
            near |= live & (near_acc | nq | npd)
            rej = live & ~acc
            if rej.any():
                w = np.maximum(0.0, q[rej] - lenience * p[rej])
                zero = w.sum(axis=1) == 0
                w[zero] = q[rej][zero]
                u2 = U(rows[rej], k, PURPOSE_RESAMPLE)
                token[rej], _ = inverse_cdf(u2, w)
                adm[rej], over = admissible_draws(u2, w)
                near[rej] |= over
                n[rej] = k
        allacc = n == gamma
        if allacc.any():
            q, nq = transformed_probs(zt[allacc, gamma], temperature, top_k, top_p)
            u2 = U(rows[allacc], gamma, PURPOSE_RESAMPLE)
            token[allacc], _ = inverse_cdf(u2, q)
            adm[allacc], over = admissible_draws(u2, q)
            near[allacc] |= over | nq

    tokens = _emit(x, n, token)
    accepted = n.copy()
    status = np.where(bad, STATUS_EDATA, STATUS_OK)
    accepted[bad] = -1
    tokens[bad] = -1
    token[bad] = -1
    near[bad] = False
    adm[bad] = -1
    return dict(accepted=accepted, tokens=tokens, next_token=token, status=status,
                near_tie=near, adm_tokens=adm, q_x=q_x, p_x=p_x, prob_near=prob_near)


def sample(logits, temperature=1.0, top_p=1.0, top_k=0, seed=0, offset=0,
           purpose=PURPOSE_DRAFT, pos0=0, uniform_fn=None):
    """Draw one token per row from the transformed distribution.

    The ordinary sampler that [SpS] Algorithm 1 (ArS) and the drafting step
    use, with the transforms of [SpS] "与标准采样方法的兼容性". logits
    [B, P, V]; token[b, j] uses U(seed, offset+b, pos0+j, purpose) and the
    inverse CDF in index order (temperature 0: argmax). A bad row (NaN,
    +inf, all -inf) gets token -1 and marks its sequence with status 4.
    Returns dict with tokens [B, P], near_tie [B, P] (top-p threshold
    near-ties, and draws with more admissible tokens than ADM_K),
    adm_tokens [B, P, ADM_K] (``admissible_draws``), status [B].
    """
    z = _f64(logits)
    B, P, V = z.shape
    U = _uniform_fn(seed, uniform_fn)
    rows = np.uint64(offset) + np.arange(B, dtype=np.uint64)
    tokens = np.full((B, P), -1, dtype=np.int64)
    adm = np.full((B, P, ADM_K), -1, dtype=np.int64)
    near = np.zeros((B, P), dtype=bool)
    bad = _bad_rows(z)
    for j in range(P):
        q, nq = transformed_probs(z[:, j], temperature, top_k, top_p)
        if temperature == 0:
            tokens[:, j] = np.argmax(q, axis=1)
            adm[:, j, 0] = tokens[:, j]
            continue
        u = U(rows, pos0 + j, purpose)
        with np.errstate(invalid="ignore"):
            qq = np.nan_to_num(q)
            tokens[:, j], _ = inverse_cdf(u, qq)
            adm[:, j], over = admissible_draws(u, qq)
        near[:, j] = nq | over
    tokens[bad] = -1
    near[bad] = False
    adm[bad] = -1
    return dict(tokens=tokens, near_tie=near, adm_tokens=adm,
                status=np.where(bad.any(axis=1), STATUS_EDATA, STATUS_OK))


# ---------------------------------------------------------------------------
# REST tree verification: [REST] "REST: 基于检索的投机解码".
# ---------------------------------------------------------------------------

def verify_tree(target, node_tokens, parent, depth, max_depth):
    """Greedy exact-match verification of a BFS pseudo-sequence.

    [REST] "REST: 基于检索的投机解码": the top-weight trie subtree is laid
    out by BFS as one pseudo-sequence scored with a tree mask; a draft token
    is accepted iff it equals the token the LLM would itself emit, so the
    output equals plain greedy decoding. Node 0 is the root (the last context
    token); row i of target [B, N, V] scores node i's children. Node i is
    accepted iff its parent is accepted and node_tokens[i] equals
    argmax(target[parent[i]]) (lowest index on ties). The deepest accepted
    node d* (lowest index on ties) ends the accepted path; the bonus token is
    argmax(target[d*]).

    Returns dict: accept_len [B] (= depth of d*), path_nodes [B, max_depth+1]
    (root..d*), tokens [B, max_depth+1] (path tokens then the bonus), bonus
    [B], status [B]. Malformed trees (parent[0] != -1, parent[i] not in
    [0, i), depth[i] != depth[parent[i]] + 1, depth[0] != 0, depth beyond
    max_depth, node token outside [0, V)) and bad rows give status 4.
    """
    z = _f64(target)
    B, N, V = z.shape
    tok = np.asarray(node_tokens, dtype=np.int64).reshape(B, N)
    par = np.asarray(parent, dtype=np.int64).reshape(B, N)
    dep = np.asarray(depth, dtype=np.int64).reshape(B, N)
    am = np.argmax(z, axis=2)
    bad = _bad_rows(z).any(axis=1)
    bad |= (par[:, 0] != -1) | (dep[:, 0] != 0)
    for i in range(1, N):
        pi = par[:, i]
        okp = (pi >= 0) & (pi < i)
        bad |= ~okp
        pc = np.clip(pi, 0, N - 1)
        bad |= dep[:, i] != dep[np.arange(B), pc] + 1
        bad |= (tok[:, i] < 0) | (tok[:, i] >= V)
    bad |= (dep > max_depth).any(axis=1)

    acc = np.zeros((B, N), dtype=bool)
    acc[:, 0] = True
    brange = np.arange(B)
    for i in range(1, N):
        pc = np.clip(par[:, i], 0, N - 1)
        acc[:, i] = acc[brange, pc] & (tok[:, i] == am[brange, pc])
    score = np.where(acc, dep, -1)
    dstar = np.argmax(score, axis=1)
    alen = dep[brange, dstar]
    W = max_depth + 1
    path = np.full((B, W), -1, dtype=np.int64)
    toks = np.full((B, W), -1, dtype=np.int64)
    bonus = am[brange, dstar].astype(np.int64)
    for b in range(B):
        if bad[b]:
            continue
        node = dstar[b]
        while node >= 0:
            path[b, dep[b, node]] = node
            node = par[b, node] if node > 0 else -1
        for j in range(alen[b]):
            toks[b, j] = tok[b, path[b, j + 1]]
        toks[b, alen[b]] = bonus[b]
    alen = np.where(bad, -1, alen)
    bonus = np.where(bad, -1, bonus)
    return dict(accept_len=alen, path_nodes=path, tokens=toks, bonus=bonus,
                status=np.where(bad, STATUS_EDATA, STATUS_OK))


# ---------------------------------------------------------------------------
# Mentor (lossy) variant: [Mentor] "导师解码", "解决优化问题".
# ---------------------------------------------------------------------------

def mentor_pi(q, p, alpha, beta):
    """Result law pi_i = p_i r_i + s_i (1 - sum_j p_j r_j) written out directly.

    [Mentor] "导师解码" (pi_i) with the KKT forms of "解决优化问题":
    r_i = min(1, q_i/(alpha p_i)), s_i = max(0, q_i/beta - p_i)/(1 - sum p r).
    Used by the tests as an independent check of the sorted prefix sums.
    alpha = 0 means r = 1 (accept all), pi = p.
    """
    q = np.asarray(q, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    if alpha == 0:
        return p.copy()
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(p > 0, np.minimum(1.0, q / (alpha * np.where(p > 0, p, 1.0))), 1.0)
    return p * r + np.maximum(0.0, q / beta - p)


def mentor_solve(q, p, kl_bound, iters=30):
    """Per-row alpha and beta of the mentor solution by bisection on alpha.

    [Mentor] "解决优化问题": r_i = min(1, q_i/(alpha p_i)) and
    s_i proportional to max(0, q_i/beta - p_i); alpha in ]0, 1] determines
    beta; the KL divergence of the result law falls as alpha grows, so
    alpha is found by bisection. The KL is KL(q || pi) (target first; the
    page's problem statement is lost, this reading is the one its prefix sums
    of q ln(q/p) support). With the indices sorted by rho = q/p ascending
    (ties: lower index first) the page's six vectorised arrays are

        cq_j = sum_{i<=j} q_i,  cp_j = sum_{i<=j} p_i,
        sq_j = sum_{i>=j} q_i,  sp_j = sum_{i>=j} p_i,
        cl_j = sum_{i<=j} q_i ln(q_i/p_i),
        g_j  = (p_j/q_j) sq_j - sp_j,

    and for a given alpha: k = #{rho < alpha}; the rejection mass is
    R = cp_{k-1} - cq_{k-1}/alpha; beta solves sum_{rho>beta}(q/beta - p) = R,
    i.e. with m the first j having g_j <= R, beta = sq_m/(R + sp_m); then

        KL(alpha) = ln(alpha) cq_{k-1} + (cl_{m-1} - cl_{k-1}) + ln(beta) sq_m

    since pi_i equals q_i/alpha below alpha, p_i between, q_i/beta above.
    Bisection: lo = 0, hi = 1, ``iters`` halvings, keep hi feasible
    (KL(mid) <= D -> hi = mid), return alpha = hi. alpha = 1 gives beta = 1
    exactly (standard speculative sampling); D = 0 gives alpha = 1 directly.

    Returns dict(alpha, beta, alpha_lo, beta_lo, alpha_hi, beta_hi, kl0,
    shortcut, near): shortcut when KL(q || p) <= D (fast path of the same
    section: accept directly); near when KL(q||p) lies within
    band = NEAR_TIE * D of D. [alpha_lo, alpha_hi] are the bisection results
    for the bounds D + band and D - band: every result a bisection can reach
    when each KL evaluation is off by at most band (the last steps of a
    bisection always sit inside the band, so the admissible answers form this
    range rather than one value). Where the range is narrower than
    NEAR_TIE * alpha, alpha itself is decided to that relative tolerance;
    where it is wider (KL nearly flat at the crossing), alpha is a near-tie.
    """
    q = np.asarray(q, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    D = float(kl_bound)
    band = NEAR_TIE * D
    with np.errstate(divide="ignore", invalid="ignore"):
        rho = np.where(p > 0, q / np.where(p > 0, p, 1.0), np.where(q > 0, np.inf, 0.0))
        qlr = np.where(q > 0, q * np.log(np.where(q > 0, rho, 1.0)), 0.0)
    kl0 = float(qlr.sum())
    near = abs(kl0 - D) <= band
    if kl0 <= D:
        return dict(alpha=0.0, beta=np.inf, kl0=kl0, shortcut=True, near=near)
    order = np.argsort(rho, kind="stable")
    qs, ps, rs, ls = q[order], p[order], rho[order], qlr[order]
    cq = np.cumsum(qs)
    cp = np.cumsum(ps)
    sq = np.cumsum(qs[::-1])[::-1]
    sp = np.cumsum(ps[::-1])[::-1]
    cl = np.cumsum(ls)
    with np.errstate(divide="ignore", invalid="ignore"):
        g = sq / rs - sp
    V = q.size

    def at(alpha):
        k = int(np.searchsorted(rs, alpha, side="left"))
        qlow = cq[k - 1] if k else 0.0
        plow = cp[k - 1] if k else 0.0
        llow = cl[k - 1] if k else 0.0
        R = plow - qlow / alpha
        m = max(int(np.searchsorted(-g, -R, side="left")), k)
        m = min(m, V - 1)
        beta = sq[m] / (R + sp[m])
        lmid = (cl[m - 1] if m else 0.0) - llow
        kl = np.log(alpha) * qlow + lmid + np.log(beta) * sq[m]
        return kl, beta

    if D == 0:
        # KL(alpha) > 0 for every alpha < 1 once KL(q||p) > 0, so D = 0 admits
        # alpha = 1 only; KL(1 - eps) ~ eps^2 sinks below fp64 rounding for
        # eps < 1e-7, so the bisection could not resolve this limit itself.
        return dict(alpha=1.0, beta=1.0, alpha_lo=1.0, beta_lo=1.0, alpha_hi=1.0, beta_hi=1.0,
                    kl0=kl0, shortcut=False, near=near)
    def bisect(bound):
        lo, hi = 0.0, 1.0
        for _ in range(iters):
            mid = 0.5 * (lo + hi)
            if at(mid)[0] <= bound:
                hi = mid
            else:
                lo = mid
        return hi

    def beta_of(a):
        return 1.0 if a == 1.0 else at(a)[1]

    alpha = bisect(D)
    # the results a bisection reaches when every KL(mid) may be off by +-band
    alpha_lo, alpha_hi = bisect(D + band), bisect(D - band)
    return dict(alpha=alpha, beta=beta_of(alpha), alpha_lo=alpha_lo, beta_lo=beta_of(alpha_lo),
                alpha_hi=alpha_hi, beta_hi=beta_of(alpha_hi), kl0=kl0, shortcut=False, near=near)


def verify_mentor(target, draft, draft_tokens, temperature=1.0, kl_bound=0.0,
                  bisect_iters=30, seed=0, offset=0, uniform_fn=None):
    """Lossy (mentor) verification.

    [Mentor] "解决优化问题" and its list of savings: a draft token passing
    the standard test u < min(1, q/p) is accepted without solving, since
    r_i >= min(1, q_i/p_i); a row with KL(q || p) <= D is accepted directly;
    otherwise alpha, beta come from ``mentor_solve`` and x is accepted iff
    u < min(1, rho_x/alpha), using the same u as the standard test. On
    rejection x ~ s, s proportional to max(0, q/beta - p), by inverse CDF in
    index order with u' = U(seed, offset+b, n, RESAMPLE). The bonus token
    (all gamma accepted) is drawn from q_gamma as in [SpS]. Temperature only
    (no top-k / top-p for this variant).

    Returns the ``verify`` dict plus alpha [B, gamma] and beta [B, gamma] for
    the decided positions k <= accepted: -1 where the standard test accepted,
    0 for the KL(q||p) <= D shortcut, the bisection result otherwise; and
    alpha_lo / alpha_hi, the range of admissible bisection results (see
    mentor_solve). A decision that differs across that range is a near-tie.
    """
    zt = _f64(target)
    B, G1, V = zt.shape
    gamma = G1 - 1
    zd = _f64(draft).reshape(B, gamma, V)
    x = np.asarray(draft_tokens, dtype=np.int64).reshape(B, gamma)
    U = _uniform_fn(seed, uniform_fn)
    rows = np.uint64(offset) + np.arange(B, dtype=np.uint64)
    bad = _bad_rows(zt).any(axis=1) | ((x < 0) | (x >= V)).any(axis=1)
    if gamma:
        bad |= _bad_rows(zd).any(axis=1)
    xs = np.clip(x, 0, V - 1)
    n = np.full(B, gamma, dtype=np.int64)
    token = np.full(B, -1, dtype=np.int64)
    adm = np.full((B, ADM_K), -1, dtype=np.int64)
    near = np.zeros(B, dtype=bool)
    alpha = np.full((B, gamma), np.nan)
    beta = np.full((B, gamma), np.nan)
    alpha_lo = np.full((B, gamma), np.nan)
    alpha_hi = np.full((B, gamma), np.nan)
    q_x = np.full((B, gamma), np.nan)
    p_x = np.full((B, gamma), np.nan)
    brange = np.arange(B)
    for k in range(gamma):
        q, _ = transformed_probs(zt[:, k], temperature)
        p, _ = transformed_probs(zd[:, k], temperature)
        q_x[:, k] = q[brange, xs[:, k]]
        p_x[:, k] = p[brange, xs[:, k]]
        u = U(rows, k, PURPOSE_ACCEPT)
        acc, rho, near_acc = accept_test(u, q_x[:, k], p_x[:, k])
        live = (n == gamma) & ~bad
        for b in np.nonzero(live)[0]:
            near[b] |= near_acc[b]
            if acc[b]:
                alpha[b, k] = -1.0
                continue
            sol = mentor_solve(q[b], p[b], kl_bound, bisect_iters)
            near[b] |= sol["near"]
            if sol["shortcut"]:
                alpha[b, k] = 0.0
                continue
            a, be = sol["alpha"], sol["beta"]
            alpha[b, k] = a
            beta[b, k] = be
            alpha_lo[b, k], alpha_hi[b, k] = sol["alpha_lo"], sol["alpha_hi"]
            thr = min(1.0, rho[b] / a)
            near[b] |= abs(u[b] - thr) <= NEAR_TIE
            near[b] |= (u[b] < min(1.0, rho[b] / sol["alpha_lo"])) != (u[b] < min(1.0, rho[b] / sol["alpha_hi"]))
            if u[b] < thr:
                continue
            u2 = U(rows[b:b + 1], k, PURPOSE_RESAMPLE)

            def weights(bb):
                w = np.maximum(0.0, q[b] / bb - p[b])
                return (w if w.sum() > 0 else q[b])[None, :]

            token[b] = inverse_cdf(u2, weights(be))[0][0]
            # admissible tokens: the band around each draw from the weights
            # of beta and of the admissible range's ends
            a_set, over = admissible_draws(u2, weights(be))
            for bb in (sol["beta_lo"], sol["beta_hi"]):
                a2, o2 = admissible_draws(u2, weights(bb))
                a_set, o3 = _merge_adm(a_set, a2)
                over |= o2 | o3
            adm[b] = a_set[0]
            near[b] |= bool(over[0])
            n[b] = k
    allacc = (n == gamma) & ~bad
    if allacc.any():
        q, _ = transformed_probs(zt[allacc, gamma], temperature)
        u2 = U(rows[allacc], gamma, PURPOSE_RESAMPLE)
        token[allacc], _ = inverse_cdf(u2, q)
        adm[allacc], over = admissible_draws(u2, q)
        near[allacc] |= over
    tokens = _emit(x, n, token)
    tokens[bad] = -1
    accepted = np.where(bad, -1, n)
    token[bad] = -1
    near[bad] = False
    adm[bad] = -1
    return dict(accepted=accepted, tokens=tokens, next_token=token,
                status=np.where(bad, STATUS_EDATA, STATUS_OK), near_tie=near, adm_tokens=adm,
                alpha=alpha, beta=beta, alpha_lo=alpha_lo, alpha_hi=alpha_hi, q_x=q_x, p_x=p_x)


# ---------------------------------------------------------------------------
# Acceptance theory and speedup formulas: [SD] "方法细节", appendix E.
# ---------------------------------------------------------------------------

def acceptance_rate(q, p):
    """beta = sum_x min(p(x), q(x)) per row.

    [SpS] appendix proof of Theorem 1 (rejection probability lines) and [SD]
    "接受率精确刻画": the probability that one draft token is accepted.
    """
    return np.minimum(np.asarray(q, np.float64), np.asarray(p, np.float64)).sum(axis=-1)


def expected_tokens(alpha, gamma):
    """E[#tokens per target call] = (1 - alpha^(gamma+1)) / (1 - alpha).

    [SD] "期望生成 token 数" (i.i.d. acceptance with rate alpha); gamma + 1
    at alpha = 1.
    """
    if alpha == 1.0:
        return gamma + 1.0
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def walltime_factor(alpha, gamma, c):
    """Expected walltime improvement (1 - alpha^(gamma+1)) / ((1-alpha)(gamma c + 1)).

    [SD] "墙钟加速因子"; c is the draft-to-target cost ratio of one call.
    """
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def ops_factor(alpha, gamma, c_hat):
    """Expected total-operations factor (1-alpha)(gamma c_hat + gamma + 1)/(1-alpha^(gamma+1)).

    [SD] "运算量分析"; c_hat is the draft-to-target cost ratio per token.
    """
    return (gamma * c_hat + gamma + 1.0) / expected_tokens(alpha, gamma)



def best_gamma(alpha, c, gamma_max):
    """The draft length in 1..gamma_max with the largest walltime factor
    (the smallest such length on ties).

    [SD] "方法细节" and its FAQ on choosing gamma: alpha is measured, c is
    the draft-to-target cost ratio, and gamma is chosen by maximising
    (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma c + 1)) numerically.
    """
    best, arg = -1.0, 1
    for g in range(1, gamma_max + 1):
        f = walltime_factor(alpha, g, c)
        if f > best:
            best, arg = f, g
    return arg


def estimate_alpha(beta):
    """alpha = E(beta): the mean of per-position acceptance probabilities.

    [SD] "接受率精确刻画": alpha is the expectation of beta = sum_x min(p, q)
    over the positions (the page measures it over 10K tokens).
    """
    b = np.asarray(beta, np.float64)
    return float(b.mean())