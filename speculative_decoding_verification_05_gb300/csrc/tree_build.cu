// REST draft-tree construction.
//
// "简单好用！北大、普林斯顿联合提出即插即用的大语言模型加速方法" (REST), section
// "REST: 基于检索的投机解码": every prefix of a retrieved continuation is a
// node of a trie weighted by how often it occurs; the heaviest nodes form the
// draft tree; its breadth-first order is the pseudo-sequence the target model
// scores, with an attention mask that restores each token's ancestry.
//
// One CTA builds one sequence's tree in shared memory, without building a
// trie. Sorted lexicographically, the candidates that share a prefix of
// length l form one run; a node is (l, k) with k the first sorted candidate
// of its run (where the common prefix with the previous candidate is shorter
// than l), its weight the multiplicities summed over the run, its children
// the nodes of depth l + 1 that start inside the run. So:
//   1. candidates into shared memory, each ended at its first -1;
//   2. bitonic sort of the candidate indices (lexicographic, index on ties;
//      each comparison made by 8 lanes reading positions in parallel);
//   3. common-prefix length with the previous sorted candidate, prefix sums
//      of the multiplicities, a sparse table of range minima of the common
//      prefixes, and every node (l, k) with its run's end e (the first later
//      candidate whose common prefix is shorter than l, found by descending
//      the table) and its weight;
//   4. the (N - 1)-th largest weight by a radix select (three 10-bit digits),
//      then a bitonic sort of the 64-bit keys of the nodes at least that heavy
//      (weight descending, length, k, then e, which (l, k) determines): the
//      first N - 1 are the chosen nodes (k order is path order);
//   5. bitonic sort of their (l, k, e) words: breadth-first positions; a
//      node's parent is the last chosen node of depth l - 1 starting at or
//      before k;
//   6. the mask: node j is node i or its ancestor iff j is no deeper than i
//      and i's first candidate lies in j's run.
// Candidate rows are stored with an odd stride, so the threads of a warp that
// read one column of different candidates hit different banks. The work is a
// few thousand integers per sequence: latency-bound, no HBM stream worth
// staging.

#include "common.cuh"
#include "specverify.h"

namespace sv {
namespace {

constexpr int TB = 1024;  // one radix bin per thread in the weight selection
constexpr int TW = TB / 32;
constexpr int kMaxC = SPEC_MAX_TREE_C;
constexpr int kMaxCL = SPEC_MAX_TREE_CL;
constexpr int kMaxN = SPEC_MAX_TREE_N;
constexpr int kLog = 10;  // 2^kLog = kMaxC

// Node key: (2^30 - 1 - weight) | l | k | e, so ascending keys rank by weight
// descending, then length, then path; breadth-first words: l | k | e.
constexpr int kKeyE = 0, kKeyK = 11, kKeyL = 22, kKeyW = 28;
SV_DEV uint32_t word_of(int l, int k, int e) {
    return ((uint32_t)l << kKeyL) | ((uint32_t)k << kKeyK) | ((uint32_t)e << kKeyE);
}

struct TreeParams {
    const int32_t* cand;
    const int32_t* counts;
    const int32_t* root;
    int B, C, L, V, N;
    int32_t* tokens;
    int32_t* parent;
    int32_t* depth;
    uint8_t* mask;
    int32_t* n_nodes;
    int32_t* status;
};

struct TreeSmem {
    int32_t tok[kMaxCL + kMaxC];  // candidate c, position l at c * LS + l (LS odd); -1 after its end
    int32_t len[kMaxC];
    int32_t cnt[kMaxC];
    int32_t ord[kMaxC];          // sorted position -> candidate
    int32_t lcp[kMaxC];          // common prefix with the previous sorted candidate
    int32_t pm[kMaxC + 1];       // exclusive prefix sums of the sorted multiplicities
    int32_t noff[kMaxC + 1];     // first node of each sorted candidate
    uint8_t mn[kLog + 1][kMaxC]; // mn[j][i] = min(lcp[i .. i + 2^j))
    uint32_t bfs[kMaxN];         // chosen words (l, k, e), breadth-first order
    union {
        unsigned long long key[kMaxCL];  // node keys (steps 3-4)
        struct {
            int32_t l[kMaxN], k[kMaxN], e[kMaxN];  // position -> depth, run start, run end
        } pos;
    } u;
    uint32_t hist[TB];           // weight selection: digit counts
    int32_t scan[TW + 1];
    int32_t sel[4];
    int32_t flag;
};

// Lexicographic order of candidates a, b on their first `l` tokens (-1 after
// a candidate's end sorts first): <0, 0, >0. LS is the row stride.
SV_DEV int cmp_prefix(const TreeSmem& s, int LS, int a, int b, int l) {
    for (int i = 0; i < l; ++i) {
        const int x = s.tok[a * LS + i], y = s.tok[b * LS + i];
        if (x != y) return x < y ? -1 : 1;
    }
    return 0;
}

// Ascending bitonic sort of n (a power of two) elements; every thread calls.
template <typename T, typename Less>
SV_DEV void bitonic(T* a, int n, Less less) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += TB) {
                const int p = i ^ j;
                if (p > i) {
                    const T x = a[i], y = a[p];
                    const bool up = (i & k) == 0;
                    if (up ? less(y, x) : less(x, y)) {
                        a[i] = y;
                        a[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Exclusive scan of a[0, n) in place, n <= 2 * TB; returns the total.
SV_DEV int block_scan(TreeSmem& s, int32_t* a, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = 2 * tid;
    const int x0 = i0 < n ? a[i0] : 0, x1 = i0 + 1 < n ? a[i0 + 1] : 0;
    const int t = x0 + x1;
    int incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < TW ? s.scan[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < TW) s.scan[lane] = wi - w;
        if (lane == 31) s.scan[TW] = wi;
    }
    __syncthreads();
    const int base = s.scan[warp] + incl - t;
    if (i0 < n) a[i0] = base;
    if (i0 + 1 < n) a[i0 + 1] = base + x0;
    const int total = s.scan[TW];
    __syncthreads();
    return total;
}

// End of the run of sorted candidates sharing the first l tokens of sorted
// candidate k: the first k2 > k with lcp[k2] < l (C if none), by jumping over
// blocks whose minimum is at least l.
SV_DEV int run_end(const TreeSmem& s, int C, int k, int l) {
    int pos = k + 1;
    for (int j = kLog; j >= 0; --j)
        if (pos + (1 << j) <= C && (int)s.mn[j][pos] >= l) pos += 1 << j;
    return pos;
}

// Inclusive scan of one value per thread over the CTA.
SV_DEV int block_incl_scan(TreeSmem& s, int v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s.scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < TW ? s.scan[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < TW) s.scan[lane] = wi - w;
    }
    __syncthreads();
    const int r = incl + s.scan[warp];
    __syncthreads();
    return r;
}

SV_DEV uint32_t weight_of(unsigned long long key) { return ((1u << 30) - 1u) - (uint32_t)(key >> kKeyW); }

// The R-th largest weight among the M node keys (1 <= R <= M), digit by digit
// from the top (three 10-bit digits of the 30-bit weights).
SV_DEV uint32_t kth_weight(TreeSmem& s, int M, int R) {
    static_assert(TB == 1024, "one bin per thread");
    const int tid = threadIdx.x;
    uint32_t prefix = 0;
    int r = R;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = 20 - 10 * pass;
        s.hist[tid] = 0u;
        __syncthreads();
        for (int o = tid; o < M; o += TB) {
            const uint32_t w = weight_of(s.u.key[o]);
            if (pass == 0 || (w >> (shift + 10)) == (prefix >> (shift + 10)))
                atomicAdd(&s.hist[(w >> shift) & 1023u], 1u);
        }
        __syncthreads();
        const int c = (int)s.hist[1023 - tid];  // thread t: digit 1023 - t (descending)
        const int incl = block_incl_scan(s, c);
        if (incl - c < r && incl >= r) {
            s.sel[0] = 1023 - tid;
            s.sel[1] = r - (incl - c);
        }
        __syncthreads();
        prefix |= (uint32_t)s.sel[0] << shift;
        r = s.sel[1];
        __syncthreads();
    }
    return prefix;
}

// Bitonic sort of the candidate indices (lexicographic, index on ties). Each
// comparison is made by a group of 8 lanes: lane r reads positions r, r + 8,
// ...; the group's first differing position decides.
SV_DEV void sort_candidates(TreeSmem& s, int C, int L, int LS, int CP) {
    constexpr int G = TB / 8;
    const int tid = threadIdx.x, r = tid & 7, g = tid >> 3;
    const int pairs = CP >> 1;
    for (int k = 2; k <= CP; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t0 = 0; t0 < pairs; t0 += G) {  // the same trip count in every lane
                const int t = t0 + g;
                const bool act = t < pairs;
                const int i = act ? (((t & ~(j - 1)) << 1) | (t & (j - 1))) : 0;  // bit j of i clear
                const int q = i + j;
                const int a = act ? s.ord[i] : 0, c = act ? s.ord[q] : 0;
                const bool real = a < C && c < C;
                int fd = L;
                if (real) {
                    for (int x = r; x < L; x += 8) {
                        if (s.tok[a * LS + x] != s.tok[c * LS + x]) {
                            fd = x;
                            break;
                        }
                    }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) fd = min(fd, __shfl_xor_sync(0xFFFFFFFFu, fd, o, 8));
                int cmp;
                if (real && fd < L)
                    cmp = s.tok[a * LS + fd] < s.tok[c * LS + fd] ? -1 : 1;
                else
                    cmp = a < c ? -1 : (a > c ? 1 : 0);
                const bool swap = (i & k) == 0 ? cmp > 0 : cmp < 0;
                if (act && r == 0 && swap) {
                    s.ord[i] = c;
                    s.ord[q] = a;
                }
            }
            __syncthreads();
        }
    }
}

SV_DEV int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

__global__ void __launch_bounds__(TB) tree_build_kernel(const __grid_constant__ TreeParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TreeSmem& s = *reinterpret_cast<TreeSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int C = p.C, L = p.L, N = p.N, LS = L | 1;
    const int b = blockIdx.x;
    const int32_t* cb = p.cand + (size_t)b * C * L;
    const int root = p.root[b];

    // 1. candidates, multiplicities, validation
    int bad = root < 0 || root >= p.V;
    for (int e = tid; e < C * L; e += TB) {
        const int t = cb[e];
        bad |= t < -1 || t >= p.V;
        const int c = e / L;
        s.tok[c * LS + (e - c * L)] = t;
    }
    for (int c = tid; c < C; c += TB) {
        const int m = p.counts ? p.counts[(size_t)b * C + c] : 1;
        bad |= m < 0 || m >= SPEC_TREE_MAX_COUNT;
        s.cnt[c] = m;
    }
    bad = __syncthreads_or(bad);
    if (!bad) {
        for (int c = tid; c < C; c += TB) {
            int n = L;
            for (int l = 0; l < L; ++l) {
                if (s.tok[c * LS + l] == -1) {
                    n = l;
                    break;
                }
            }
            s.len[c] = n;
            for (int l = n; l < L; ++l) s.tok[c * LS + l] = -1;
        }
        const int CP = pow2_at_least(C);
        for (int i = tid; i < CP; i += TB) s.ord[i] = i;  // CP <= kMaxC (a power of two)
        __syncthreads();

        // 2. candidates in lexicographic order
        sort_candidates(s, C, L, LS, CP);

        // 3. common prefixes, multiplicity sums, nodes
        for (int k = tid; k < C; k += TB) {
            const int a = s.ord[k];
            int lc = 0;
            if (k > 0) {
                const int pr = s.ord[k - 1];
                while (lc < L && s.tok[pr * LS + lc] == s.tok[a * LS + lc] && s.tok[a * LS + lc] != -1) ++lc;
            }
            s.lcp[k] = lc;
            s.mn[0][k] = (uint8_t)lc;
            s.pm[k] = s.cnt[a];
            s.noff[k] = max(0, s.len[a] - lc);
        }
        __syncthreads();
        const int wsum = block_scan(s, s.pm, C);
        const int M = block_scan(s, s.noff, C);
        if (tid == 0) {
            s.pm[C] = wsum;
            s.noff[C] = M;
        }
        for (int j = 1; (1 << j) <= C; ++j) {
            __syncthreads();
            const int h = 1 << (j - 1);
            for (int i = tid; i + (1 << j) <= C; i += TB) s.mn[j][i] = min(s.mn[j - 1][i], s.mn[j - 1][i + h]);
        }
        __syncthreads();
        for (int k = tid; k < C; k += TB) {
            const int a = s.ord[k];
            int o = s.noff[k];
            for (int l = s.lcp[k] + 1; l <= s.len[a]; ++l, ++o) {
                const int e = run_end(s, C, k, l);
                const uint32_t w = (uint32_t)(s.pm[e] - s.pm[k]);  // < 2^30
                s.u.key[o] = ((unsigned long long)((1u << 30) - 1u - w) << kKeyW) | word_of(l, k, e);
            }
        }
        __syncthreads();

        // 4. the heaviest N - 1 nodes: only those at least as heavy as the
        // (N - 1)-th are sorted
        int Mk = M;
        if (M > N - 1) {
            const uint32_t tau = kth_weight(s, M, N - 1);
            constexpr int kPer = kMaxCL / TB;
            unsigned long long mine[kPer];
            bool keep[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int o = tid + u * TB;
                keep[u] = o < M;
                if (keep[u]) {
                    mine[u] = s.u.key[o];
                    keep[u] = weight_of(mine[u]) >= tau;
                }
            }
            if (tid == 0) s.sel[2] = 0;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < kPer; ++u)
                if (keep[u]) s.u.key[atomicAdd(&s.sel[2], 1)] = mine[u];
            __syncthreads();
            Mk = s.sel[2];
        }
        const int MP = pow2_at_least(max(Mk, 1));
        for (int i = Mk + tid; i < MP; i += TB) s.u.key[i] = ~0ull;
        __syncthreads();
        bitonic(s.u.key, MP, [](unsigned long long x, unsigned long long y) { return x < y; });
        const int S = min(N - 1, M);
        const int SP = pow2_at_least(max(S, 1));
        for (int i = tid; i < SP; i += TB)
            s.bfs[i] = i < S ? (uint32_t)(s.u.key[i] & ((1ull << kKeyW) - 1)) : 0xFFFFFFFFu;
        __syncthreads();

        // 5. breadth-first positions, parents
        bitonic(s.bfs, SP, [](uint32_t x, uint32_t y) { return x < y; });
        for (int q = tid; q < N; q += TB) {
            int32_t tk = -1, pa = -1, de = -1;
            if (q == 0) {
                tk = root;
                de = 0;
                s.u.pos.l[0] = 0;
                s.u.pos.k[0] = 0;
                s.u.pos.e[0] = C;
            } else if (q <= S) {
                const uint32_t w = s.bfs[q - 1];
                const int l = (int)(w >> kKeyL), k = (int)((w >> kKeyK) & 0x7FFu), e = (int)(w & 0x7FFu);
                tk = s.tok[s.ord[k] * LS + l - 1];
                de = l;
                pa = 0;
                if (l > 1) {
                    // the last chosen word <= (l - 1, k, any e)
                    const uint32_t want = word_of(l - 1, k, 0x7FF);
                    int lo = 0, hi = q - 1;  // bfs[q - 1] > want
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (s.bfs[mid] <= want)
                            lo = mid + 1;
                        else
                            hi = mid;
                    }
                    pa = lo;  // position of bfs[lo - 1] is lo
                }
                s.u.pos.l[q] = l;
                s.u.pos.k[q] = k;
                s.u.pos.e[q] = e;
            }
            const size_t o = (size_t)b * N + q;
            if (SV_IN_SEQ(o, (long long)p.B * p.N, p.status, b)) {
                p.tokens[o] = tk;
                p.parent[o] = pa;
                p.depth[o] = de;
            }
        }
        if (tid == 0) {
            p.n_nodes[b] = S + 1;
            if (p.status) p.status[b] = kOk;
            s.flag = S;
        }
        __syncthreads();
    } else {
        for (int q = tid; q < N; q += TB) {
            const size_t o = (size_t)b * N + q;
            p.tokens[o] = -1;
            p.parent[o] = -1;
            p.depth[o] = -1;
        }
        if (tid == 0) {
            p.n_nodes[b] = -1;
            if (p.status) p.status[b] = kEData;
            s.flag = -1;
        }
        __syncthreads();
    }

    // 6. the tree attention mask
    if (!p.mask) return;
    const int S = s.flag;
    uint8_t* mb = p.mask + (size_t)b * N * N;
    auto bit = [&](int i, int j) -> uint32_t {
        if (i > S || j > S) return 0u;
        if (j == 0) return 1u;
        const int ki = s.u.pos.k[i];
        return (uint32_t)(s.u.pos.l[j] <= s.u.pos.l[i] && s.u.pos.k[j] <= ki && ki < s.u.pos.e[j]);
    };
    if ((N & 3) == 0 && ((uintptr_t)mb & 3) == 0) {
        uint32_t* mw = reinterpret_cast<uint32_t*>(mb);
        const int words = N * N / 4;
        for (int w = tid; w < words; w += TB) {
            const int e = 4 * w, i = e / N, j = e - i * N;
            mw[w] = bit(i, j) | (bit(i, j + 1) << 8) | (bit(i, j + 2) << 16) | (bit(i, j + 3) << 24);
        }
    } else {
        for (int e = tid; e < N * N; e += TB) {
            const int i = e / N;
            mb[e] = (uint8_t)bit(i, e - i * N);
        }
    }
}

}  // namespace

size_t tree_build_smem_bytes() { return sizeof(TreeSmem); }

cudaError_t launch_tree_build(const int32_t* cand, const int32_t* counts, const int32_t* root, int B, int C,
                              int L, int V, int N, int32_t* tokens, int32_t* parent, int32_t* depth,
                              uint8_t* mask, int32_t* n_nodes, int32_t* status, cudaStream_t stream) {
    TreeParams p;
    p.cand = cand;
    p.counts = counts;
    p.root = root;
    p.B = B;
    p.C = C;
    p.L = L;
    p.V = V;
    p.N = N;
    p.tokens = tokens;
    p.parent = parent;
    p.depth = depth;
    p.mask = mask;
    p.n_nodes = n_nodes;
    p.status = status;
    const int smem = (int)sizeof(TreeSmem);
    cudaError_t e = cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    tree_build_kernel<<<B, TB, smem, stream>>>(p);
    return cudaGetLastError();
}

SV_DEBUG_READER(tree_build)

}  // namespace sv
