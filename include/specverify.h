/*
 * specverify.h - C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * The library turns target logits over gamma+1 positions and draft logits over
 * gamma positions into accepted tokens, as the pages define it:
 *
 *   [SpS]    "Accelerating Large Language Model Decoding with Speculative
 *            Sampling" (notes on Chen et al., 2023), section "改进的拒绝采样"
 *            (accept x with probability min(1, q(x)/p(x)) left to right, stop
 *            at the first rejection, resample from (q-p)+; all accepted ->
 *            one bonus token from the last target row) and
 *            "与标准采样方法的兼容性" (temperature / top-k / nucleus applied
 *            to the probabilities first).
 *   [SD]     "Fast Inference from Transformers via Speculative Decoding"
 *            write-up, "标准化采样框架" (argmax is temperature 0).
 *   [REST]   "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法",
 *            "REST: 基于检索的投机解码" (greedy exact-match verification of a
 *            BFS pseudo-sequence of a draft trie).
 *   [Mentor] "推测解码的一种最优有损变体", "解决优化问题" (lossy variant: per
 *            row alpha by bisection so that r_i = min(1, q_i/(alpha p_i)) and
 *            s_i ~ max(0, q_i/beta - p_i) meet a KL bound D).
 *
 * Conventions shared by every entry point:
 *
 *  - q is the target distribution, p the draft distribution.
 *  - All tensor arguments are DEVICE pointers owned by the caller, row-major
 *    and contiguous (innermost dimension V). Logit pointers need only be
 *    aligned to their element size; rows of any length are handled.
 *  - Every call is asynchronous: it validates its arguments on the host,
 *    enqueues its kernels on `stream` and returns. Outputs are valid once the
 *    stream has reached that point.
 *  - Host-detectable errors (null pointers, sizes out of range, bad sampling
 *    parameters, workspace too small or misaligned) return SPEC_EINVAL and
 *    enqueue nothing. A failed kernel launch returns SPEC_ECUDA.
 *  - Errors found in the data on the device are reported per sequence in
 *    `status[b]` (when `status` is not NULL): SPEC_EDATA for a logit row that
 *    holds NaN or +inf or only -inf, a draft token outside [0, V), or a
 *    malformed tree; that sequence's outputs are then all -1. -inf alone is
 *    an ordinary zero-probability logit. SPEC_ETIMEOUT: a bounded device
 *    wait gave up. Kernels never wait on other CTAs (every hand-off between
 *    CTAs is a last-arriver counter); only the warps of one CTA of the
 *    shared-memory row path wait on one another (bounded, about a second),
 *    and when one such wait gives up, the rows that CTA had left are
 *    reported with SPEC_ETIMEOUT (outputs -1).
 *  - Workspace: a device buffer of at least the size the matching
 *    *_workspace_size() function returns, 256-byte aligned, owned by the
 *    caller. Its content on entry does not matter: each call clears the small
 *    control region it needs (one cudaMemsetAsync on `stream`) before its
 *    kernels. Calls that share a workspace must not overlap on the GPU.
 *  - Randomness: Philox-4x32-10 (Salmon et al., SC'11) with
 *    key = (seed lo, seed hi), counter = (row lo, row hi, position, purpose),
 *    row = offset + b; u = ((word0 >> 9) + 0.5) * 2^-23. The acceptance test
 *    at position k uses purpose SPEC_PURPOSE_ACCEPT, the resampled or bonus
 *    token at position n uses SPEC_PURPOSE_RESAMPLE. Calls with the same
 *    seed, offset and inputs return the same tokens.
 *  - Sampling transforms (both q and p): temperature T, then top-k (keep
 *    every logit >= the k-th largest, ties kept), then top-p (keep the
 *    logits >= tau, tau the largest logit value whose cumulative mass in the
 *    top-k renormalised distribution reaches top_p; the crossing value and
 *    its ties are kept). T = 0 is argmax (lowest index on ties).
 *    top_k = 0 (or >= V) and top_p = 1 switch those transforms off.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,   /* bad argument; nothing was enqueued */
    SPEC_ECUDA = 2,    /* a CUDA launch or attribute call failed */
    SPEC_ETIMEOUT = 3, /* (status[] only) a bounded device wait gave up */
    SPEC_EDATA = 4,    /* (status[] only) bad logits, tokens or tree */
    SPEC_EBOUNDS = 5   /* (status[] only, debug builds) an index check failed; the access was skipped */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* temperature >= 0 (0 = argmax); 0 < top_p <= 1 (1 = off); top_k >= 0 (0 = off). */
typedef struct {
    float temperature;
    float top_p;
    int32_t top_k;
} spec_sampling;

/* A cudaStream_t. NULL is the legacy default stream. */
typedef struct CUstream_st* spec_stream;

enum {
    SPEC_PURPOSE_ACCEPT = 0,
    SPEC_PURPOSE_RESAMPLE = 1,
    SPEC_PURPOSE_DRAFT = 2
};

/* Size limits checked by every entry point. */
enum {
    SPEC_MAX_V = 262144,      /* vocabulary size */
    SPEC_MAX_GAMMA = 255,     /* draft length */
    SPEC_MAX_TREE_N = 1024,   /* tree nodes, root included */
    SPEC_MAX_BISECT = 64,     /* mentor bisection iterations */
    SPEC_MAX_TREE_C = 1024,   /* tree construction: candidates per sequence */
    SPEC_MAX_TREE_L = 32,     /*                    tokens per candidate */
    SPEC_MAX_TREE_CL = 4096,  /*                    candidates x tokens */
    SPEC_TREE_MAX_COUNT = 1 << 20  /* multiplicities are below this */
};

/* ------------------------------------------------------------------------
 * spec_verify - batched modified rejection sampling ([SpS] "改进的拒绝采样",
 * "与标准采样方法的兼容性"; [SD] "标准化采样框架" for temperature 0).
 *
 *   target        [B, gamma+1, V] logits of the target model
 *   draft         [B, gamma, V] logits of the draft model; may be NULL when
 *                 sampling.temperature == 0 (argmax verification reads only
 *                 the target rows)
 *   dtype         element type of both logit tensors
 *   draft_tokens  [B, gamma] int32 draft tokens x_k
 *   B, gamma, V   1 <= B <= 2^24, 1 <= gamma <= SPEC_MAX_GAMMA, 1 <= V <= SPEC_MAX_V
 *   sampling      transform applied to q and p before the test
 *   seed, offset  Philox key and row base (row = offset + b)
 * Outputs (device, written for every b):
 *   accepted      [B] number of accepted draft tokens n in [0, gamma]
 *   tokens        [B, gamma+1] x_0..x_{n-1}, then the resampled (n < gamma)
 *                 or bonus (n = gamma) token, then -1
 *   next_token    [B] the resampled or bonus token
 *   status        [B] SPEC_OK / SPEC_EDATA / SPEC_ETIMEOUT; may be NULL
 *   probs_dbg     [B, gamma, 2] (q(x_k), p(x_k)) as computed on the device,
 *                 for every position (also those after the first
 *                 rejection); may be NULL
 *   workspace     >= spec_verify_workspace_size(B, gamma, V, dtype) bytes
 * ---------------------------------------------------------------------- */
size_t spec_verify_workspace_size(int B, int gamma, int V, spec_dtype dtype);

spec_status spec_verify(const void* target, const void* draft, spec_dtype dtype,
                        const int32_t* draft_tokens, int B, int gamma, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset,
                        int32_t* accepted, int32_t* tokens, int32_t* next_token,
                        int32_t* status, float* probs_dbg,
                        void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_verify_lenient - lenient verification ([SD] "方法细节", the lenience
 * extension of its appendix F): the draft probability is scaled by
 * `lenience` = l in ]0, 1] before the comparison, so x_k is accepted with
 * probability min(1, q(x)/(l p(x))), and a rejection resamples from
 * norm(max(0, q - l p)) (from q if that vanishes). No token is emitted with
 * probability above q(x)/l; l = 1 is spec_verify exactly. Arguments,
 * outputs, workspace and errors as spec_verify (l outside ]0, 1] or not
 * finite: SPEC_EINVAL). Temperature 0 ignores l (same decisions).
 * ---------------------------------------------------------------------- */
spec_status spec_verify_lenient(const void* target, const void* draft, spec_dtype dtype,
                                const int32_t* draft_tokens, int B, int gamma, int V,
                                spec_sampling sampling, float lenience, uint64_t seed, uint64_t offset,
                                int32_t* accepted, int32_t* tokens, int32_t* next_token,
                                int32_t* status, float* probs_dbg,
                                void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_verify_tree - greedy exact-match verification of a REST draft tree
 * ([REST] "REST: 基于检索的投机解码").
 *
 *   target        [B, N, V] logits; row i scores the children of node i
 *   node_tokens   [B, N] int32 token of each node (node 0, the root, is the
 *                 last context token and is not verified)
 *   parent        [B, N] int32; parent[0] = -1, 0 <= parent[i] < i (BFS order)
 *   depth         [B, N] int32; depth[0] = 0, depth[i] = depth[parent[i]] + 1
 *   B, N, V       1 <= N <= SPEC_MAX_TREE_N; 0 <= max_depth < N
 * A node is accepted iff its parent is accepted and its token equals the
 * argmax (lowest index on ties) of its parent's row; the deepest accepted
 * node d* (lowest index on ties) ends the path.
 * Outputs:
 *   accept_len    [B] depth of d*
 *   path_nodes    [B, max_depth+1] node indices root..d*, then -1
 *   tokens        [B, max_depth+1] tokens of path nodes 1..d*, then the bonus
 *                 token argmax(target[d*]), then -1
 *   bonus         [B] argmax(target[d*])
 *   status        [B] (NULL allowed); depth > max_depth is SPEC_EDATA
 * ---------------------------------------------------------------------- */
size_t spec_verify_tree_workspace_size(int B, int N, int V, spec_dtype dtype);

spec_status spec_verify_tree(const void* target, spec_dtype dtype,
                             const int32_t* node_tokens, const int32_t* parent,
                             const int32_t* depth, int B, int N, int V, int max_depth,
                             int32_t* accept_len, int32_t* path_nodes, int32_t* tokens,
                             int32_t* bonus, int32_t* status,
                             void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_tree_build - the REST draft tree of each sequence from its retrieved
 * continuations ([REST] "REST: 基于检索的投机解码"): every prefix of a
 * candidate is a trie node whose weight is how often the prefix occurs (the
 * sum of the multiplicities of the candidates that start with it); the N - 1
 * nodes ranked first by (weight descending, length ascending, token path
 * lexicographically ascending) form the draft tree, which is closed under
 * taking parents; its breadth-first order (a node's children by ascending
 * token) is the pseudo-sequence spec_verify_tree takes, and `mask` is its
 * tree attention mask.
 *
 *   candidates    [B, C, L] int32; a candidate ends at its first -1; every
 *                 entry must be -1 or a token in [0, V)
 *   counts        [B, C] int32 multiplicities in [0, SPEC_TREE_MAX_COUNT);
 *                 NULL: every candidate counts once
 *   root_token    [B] int32 in [0, V): the last context token (node 0)
 *   B, C, L, V, N 1 <= B <= 2^24, 1 <= C <= SPEC_MAX_TREE_C,
 *                 1 <= L <= SPEC_MAX_TREE_L, C * L <= SPEC_MAX_TREE_CL,
 *                 1 <= V, 2 <= N <= SPEC_MAX_TREE_N
 * Outputs (device, written for every b; all pointers 4-byte aligned except
 * mask):
 *   node_tokens   [B, N] int32 token of each node, root first
 *   parent        [B, N] int32, parent[0] = -1, 0 <= parent[i] < i
 *   depth         [B, N] int32, depth[0] = 0
 *                 (positions n_nodes[b] .. N-1 hold -1 in all three)
 *   mask          [B, N, N] uint8, mask[b][i][j] = 1 iff node j is node i or
 *                 one of its ancestors (rows from n_nodes[b] on are zero);
 *                 NULL allowed
 *   n_nodes       [B] int32: 1 + the number of chosen nodes, at most N (fewer
 *                 when the candidates have fewer distinct prefixes)
 *   status        [B] SPEC_OK, or SPEC_EDATA for an entry, multiplicity or
 *                 root token out of range (that sequence's outputs are -1 and
 *                 its mask rows zero); NULL allowed
 * No workspace: each sequence is built in one CTA's shared memory. Invalid
 * sizes or NULL required pointers: SPEC_EINVAL, nothing enqueued.
 * ---------------------------------------------------------------------- */
spec_status spec_tree_build(const int32_t* candidates, const int32_t* counts, const int32_t* root_token,
                            int B, int C, int L, int V, int N,
                            int32_t* node_tokens, int32_t* parent, int32_t* depth, uint8_t* mask,
                            int32_t* n_nodes, int32_t* status, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_acceptance_rate - the probability that each draft position is
 * accepted ([SD] "方法细节", 接受率精确刻画; [SpS] appendix proof of Theorem
 * 1): beta[b, k] = sum_x min(q_k(x), p_k(x)) for target row k and draft row
 * k (k < gamma) of sequence b, under the same temperature / top-k / top-p
 * transform as spec_verify. The mean of beta over positions estimates the
 * acceptance rate alpha that spec_expected_tokens and spec_best_gamma take.
 *
 * Arguments as spec_verify (no draft tokens are needed); temperature must be
 * > 0 (at temperature 0, beta is 1 where the two argmaxes agree and 0
 * elsewhere; that case returns SPEC_EINVAL).
 *   beta          [B, gamma] float (device); NaN for a pair with a non-finite
 *                 row
 *   status        [B] SPEC_OK / SPEC_EDATA; NULL allowed
 *   workspace     >= spec_verify_workspace_size(B, gamma, V, dtype) bytes
 * ---------------------------------------------------------------------- */
spec_status spec_acceptance_rate(const void* target, const void* draft, spec_dtype dtype, int B, int gamma,
                                 int V, spec_sampling sampling, float* beta, int32_t* status,
                                 void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * The alpha / gamma planner ([SD] "方法细节": 期望生成 token 数, 墙钟加速因子,
 * 运算量分析, and its FAQ on choosing gamma). Host arithmetic, no GPU:
 *   spec_expected_tokens  E[#tokens per target call] =
 *                         (1 - alpha^(gamma+1)) / (1 - alpha), gamma + 1 at
 *                         alpha = 1 (i.i.d. acceptance with rate alpha)
 *   spec_walltime_factor  spec_expected_tokens / (gamma c + 1), c the cost of
 *                         one draft call relative to one target call
 *   spec_ops_factor       (gamma c_hat + gamma + 1) / spec_expected_tokens,
 *                         c_hat the draft-to-target cost ratio per token
 *   spec_best_gamma       the gamma in 1..gamma_max with the largest
 *                         walltime factor (the smallest on ties)
 * alpha must lie in [0, 1], gamma >= 0, c and c_hat finite and >= 0;
 * otherwise the factors are NaN and spec_best_gamma returns -1.
 * ---------------------------------------------------------------------- */
double spec_expected_tokens(double alpha, int gamma);
double spec_walltime_factor(double alpha, int gamma, double c);
double spec_ops_factor(double alpha, int gamma, double c_hat);
int spec_best_gamma(double alpha, double c, int gamma_max);

/* ------------------------------------------------------------------------
 * spec_verify_mentor - lossy "mentor" verification ([Mentor] "导师解码",
 * "解决优化问题").
 *
 * Arguments as spec_verify, with temperature > 0 and no top-k / top-p, plus:
 *   kl_bound      D >= 0: bound on KL(q || pi) for the result law pi
 *   bisect_iters  bisection steps on alpha in ]0, 1] (1..SPEC_MAX_BISECT)
 *   alpha_out     [B, gamma] (NULL allowed): for the decided positions
 *                 k <= accepted[b]: -1 where the standard test u < min(1, q/p)
 *                 accepted, 0 where KL(q||p) <= D accepted directly,
 *                 otherwise the bisection's alpha. NaN after the first
 *                 rejection and for sequences with status SPEC_EDATA (those
 *                 positions are never decided, so nothing is solved there).
 *   beta_out      [B, gamma] (NULL allowed): beta for solved positions, 0 for
 *                 the two acceptance codes, NaN where alpha_out is NaN
 * A position that fails the standard test is accepted iff
 * u < min(1, q(x)/(alpha p(x))) with the same u; on rejection the token is
 * drawn from max(0, q/beta - p). The bonus token comes from q_gamma.
 * D = 0 reproduces spec_verify exactly.
 * ---------------------------------------------------------------------- */
size_t spec_verify_mentor_workspace_size(int B, int gamma, int V, spec_dtype dtype);

spec_status spec_verify_mentor(const void* target, const void* draft, spec_dtype dtype,
                               const int32_t* draft_tokens, int B, int gamma, int V,
                               float temperature, float kl_bound, int bisect_iters,
                               uint64_t seed, uint64_t offset,
                               int32_t* accepted, int32_t* tokens, int32_t* next_token,
                               int32_t* status, float* alpha_out, float* beta_out,
                               float* probs_dbg,
                               void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_sample - draw one token per row from the transformed distribution:
 * the ordinary sampler of [SpS] Algorithm 1 (ArS) and of the drafting step.
 *
 *   logits        [B, P, V], 1 <= P <= 1024
 *   tokens_out    [B, P] int32; token (b, j) uses
 *                 u = U(seed, offset + b, pos0 + j, purpose) and the inverse
 *                 CDF in index order (temperature 0: argmax)
 *   status        [B] (NULL allowed)
 * ---------------------------------------------------------------------- */
size_t spec_sample_workspace_size(int B, int P, int V, spec_dtype dtype);

spec_status spec_sample(const void* logits, spec_dtype dtype, int B, int P, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset,
                        uint32_t pos0, uint32_t purpose,
                        int32_t* tokens_out, int32_t* status,
                        void* workspace, size_t ws_bytes, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_philox_uniform - the library's uniforms, for checking a host copy of
 * the generator: out[i] = U(seed, row0 + i, position, purpose), i < n, with
 * U as defined at the top of this header. out: device float[n]; 1 <= n <= 2^30.
 * ---------------------------------------------------------------------- */
spec_status spec_philox_uniform(uint64_t seed, uint64_t row0, uint32_t position, uint32_t purpose,
                                int n, float* out, spec_stream stream);

/* ------------------------------------------------------------------------
 * spec_verify_noalloc - spec_verify without a workspace argument, for
 * callers that cannot allocate device memory when they verify (an engine
 * plugin whose framework owns all device allocations, a server with a
 * device memory budget fixed at start-up, a C caller without a device
 * allocator). The pages have no counterpart: this is a deployment variant of
 * spec_verify, with the same arguments (minus workspace / ws_bytes), the
 * same kernels and the same outputs.
 *
 * Its scratch memory is a fixed array of SPEC_NOALLOC_SCRATCH_BYTES in the
 * library's device image, held by every GPU that loads the library until the
 * process exits. Returns SPEC_EINVAL when the call would need more scratch
 * than that (spec_verify_workspace_size(B, gamma, V, dtype) >
 * SPEC_NOALLOC_SCRATCH_BYTES). It never calls cudaMalloc, cudaFree or any
 * allocating routine. The first call on a device looks the array's device
 * address up (cudaGetSymbolAddress) and caches it for that device. With
 * CUDA's lazy module loading (the default since CUDA 12.2) that first call is
 * also the moment the array's module is loaded and its
 * SPEC_NOALLOC_SCRATCH_BYTES of device memory are committed, so a caller with
 * a fixed device budget should make one call per device at start-up, before
 * any stream capture; later calls take no device memory. The cached address
 * belongs to the device's current context: resetting the device
 * (cudaDeviceReset, or destroying the primary context) after the first call
 * is not supported. All calls share the array and it keeps the last call's
 * contents (each call clears what must start at zero); calls that overlap on
 * the GPU race on it.
 * ---------------------------------------------------------------------- */
enum { SPEC_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024 };

spec_status spec_verify_noalloc(const void* target, const void* draft, spec_dtype dtype,
                                const int32_t* draft_tokens, int B, int gamma, int V,
                                spec_sampling sampling, uint64_t seed, uint64_t offset,
                                int32_t* accepted, int32_t* tokens, int32_t* next_token,
                                int32_t* status, float* probs_dbg, spec_stream stream);

/* Human-readable name of a status code (static storage). */
const char* spec_status_string(spec_status s);

/* The last CUDA error string recorded by a call that returned SPEC_ECUDA on
 * this host thread (static per-thread storage; "" if none). */
const char* spec_last_cuda_error(void);

/* Debug builds. The library built with -DSPEC_DEBUG (build.py's debug
 * library, libspecverify_debug.so) checks the indices its kernels compute
 * against the extent of the array each addresses, where a memory checker
 * cannot be run: a failed check skips the access, counts the failure and,
 * where the kernel knows the sequence, sets its status to SPEC_EBOUNDS
 * (nothing traps). spec_debug_build returns 1 for that library, 0 for the
 * release one. spec_debug_failures returns the number of failed checks on the
 * current device since the library was loaded (0 in release builds) and, when
 * `line` is not NULL, the source line of the first one (0 if none); it waits
 * for the device's queued work to finish; -1 on a CUDA error. */
int spec_debug_build(void);
int spec_debug_failures(int* line);

/* Debug builds only: the shared-memory row kernel of later calls on the
 * current device withholds the bulk copy of the j-th row its first CTA takes
 * (j < 0: none, the default). Nothing then completes that buffer's
 * barrier: the CTA's bounded waits give up (within about a second), its rows
 * from that one on are reported SPEC_ETIMEOUT in status[] (outputs -1), the
 * other CTAs' rows are verified as usual, and the device stays usable. It
 * exercises the timeout path without a fault. Returns 0; -1 in release
 * builds (nothing is changed) or on a CUDA error. */
int spec_debug_withhold_copy(int j);

/* Library ABI version (major * 100 + minor). */
int spec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
