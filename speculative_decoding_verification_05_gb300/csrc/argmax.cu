// Row-argmax kernel for greedy verification.
//
// Used by three entry points:
//  * spec_verify at temperature 0 ("Fast Inference from Transformers via
//    Speculative Decoding" write-up, "标准化采样框架": argmax is one of the
//    standard samplers): accept x_k iff it is the target argmax of row k,
//    emit the argmax of the first mismatching (or last) row;
//  * spec_verify_tree (REST, "REST: 基于检索的投机解码"): a node is accepted
//    iff its token is the argmax of its parent's row and its parent is
//    accepted; the deepest accepted node ends the path;
//  * spec_sample at temperature 0.
//
// The rows of all sequences form one flattened [rows, V] range that is cut
// into equal contiguous chunks, one per CTA, so every SM streams the same
// number of bytes whatever B, N or V are. Each row segment's argmax (lowest
// index on ties) is folded into a packed 64-bit word (key << 32 | ~index) with
// one atomicMax per warp and segment (no CTA barrier between segments); the
// CTA that completes the last element of a sequence (element counter, no
// waiting) resolves that sequence and clears its workspace.

#include "common.cuh"

namespace sv {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kMaxN = 1024;

struct Best {
    float v;
    int i;  // -1: empty
};

SV_DEV void take(Best& b, float x, int i) {
    if (x > b.v || b.i < 0) {
        b.v = x;
        b.i = i;
    }
}

SV_DEV Best better(Best a, Best b) {
    if (a.i < 0) return b;
    if (b.i < 0) return a;
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

SV_DEV Best warp_best(Best b) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        Best c;
        c.v = __shfl_xor_sync(0xFFFFFFFFu, b.v, o);
        c.i = __shfl_xor_sync(0xFFFFFFFFu, b.i, o);
        b = better(b, c);
    }
    return b;
}

struct SharedA {
    int am[kMaxN];
    int bad[kMaxN];
    int tok[kMaxN];
    int par[kMaxN];
    int dep[kMaxN];
    int path[kMaxN];   // tree: accepted flags
    int pn[kMaxN];     // tree: path node at each depth
    int bi[8];
};

// NaN-propagating maximum of the logits of one 16-byte vector.
SV_DEV float vec_max(const uint4& v, float) {
    float a, b, r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(a) : "f"(__uint_as_float(v.x)), "f"(__uint_as_float(v.y)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(b) : "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

SV_DEV float vec_max(const uint4& v, bf16_t) {
    uint32_t a, b, m;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(__uint_as_float(m << 16)), "f"(__uint_as_float(m & 0xFFFF0000u)));
    return r;
}

template <typename E>
SV_DEV void segment(const ArgmaxParams& p, long long r, int i0, int i1) {
    using T = VecTraits<E>;
    constexpr int es = sizeof(E);
    constexpr int VE = T::kN;
    const int tid = threadIdx.x, lane = tid & 31;
    const E* row = reinterpret_cast<const E*>(p.logits) + r * (long long)p.V;
    Best best{-INFINITY, -1};
    bool bad = false;
    const uintptr_t a = (uintptr_t)(row + i0);
    const int head = min(i1 - i0, (int)(((16 - (a & 15)) & 15) / es));
    for (int t = tid; t < head; t += NT) {
        const float x = T::load1(row + i0 + t);
        bad |= !(x < INFINITY);
        take(best, x, i0 + t);
    }
    const int base = i0 + head;
    const int nb = (i1 - base) / VE;
    const uint4* vp = reinterpret_cast<const uint4*>(row + base);
    constexpr int U = 4;  // 16-byte vectors in flight per thread
    for (int j = tid; j < nb; j += NT * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (j + u * NT < nb) v[u] = ld_stream_v4(vp + j + u * NT);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j + u * NT < nb) {
                // the vector's maximum decides; the index is looked up only when it
                // beats this thread's best (vectors come in increasing index order,
                // so equal values keep the lower index)
                const float vm = vec_max(v[u], E{});
                bad |= !(vm < INFINITY);
                if (vm > best.v || best.i < 0) {
                    float x[VE];
                    T::unpack(v[u], x);
                    int e0 = VE - 1;
#pragma unroll
                    for (int e = VE - 1; e >= 0; --e)
                        if (x[e] == vm) e0 = e;
                    best.v = vm;
                    best.i = base + (j + u * NT) * VE + e0;
                }
            }
        }
    }
    for (int t = base + nb * VE + tid; t < i1; t += NT) {
        const float x = T::load1(row + t);
        bad |= !(x < INFINITY);
        take(best, x, t);
    }
    // each warp folds its best into the row's word: no CTA barrier, so the
    // warps run on into the next segment independently
    best = warp_best(best);
    const int wbad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
        if (best.i >= 0) {
            const unsigned long long packed =
                ((unsigned long long)f32_key(best.v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)best.i);
            if (SV_IN(r, (long long)p.B * p.rows_per_b)) atomicMax(&p.rowbest[r], packed);
        }
        if (wbad && SV_IN(r, (long long)p.B * p.rows_per_b)) atomicOr(&p.rowbad[r], 1u);
    }
}

// Resolve sequence b from the per-row argmaxes; the whole CTA takes part.
SV_DEV void resolve(const ArgmaxParams& p, SharedA& s, int b) {
    const int tid = threadIdx.x;
    const int R = p.rows_per_b;
    const long long base = (long long)b * R;
    for (int i = tid; i < R; i += NT) {
        if (!SV_IN(i, kMaxN)) continue;
        const unsigned long long w = __ldcg(&p.rowbest[base + i]);
        const unsigned bad = __ldcg(&p.rowbad[base + i]);
        s.am[i] = (int)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFull));
        // a row whose maximum is -inf (all -inf) or whose key is below (NaN) is bad
        s.bad[i] = (bad != 0) || (uint32_t)(w >> 32) <= kKeyNegInf;
        p.rowbest[base + i] = 0ull;
        p.rowbad[base + i] = 0u;
    }
    __syncthreads();

    if (p.mode == kArgVerify) {
        const int gamma = R - 1;
        for (int i = tid; i < gamma; i += NT) {
            const int x = p.draft_tokens[(size_t)b * gamma + i];
            s.tok[i] = x;
            if (x < 0 || x >= p.V) s.bad[i] = 1;
        }
        __syncthreads();
        if (tid == 0) {
            int anybad = 0, n = gamma;
            for (int i = 0; i < R; ++i) anybad |= s.bad[i];
            for (int i = 0; i < gamma; ++i)
                if (s.tok[i] != s.am[i]) {
                    n = i;
                    break;
                }
            s.bi[0] = n;
            s.bi[1] = anybad;
            p.out0[b] = anybad ? -1 : n;
            p.out2[b] = anybad ? -1 : s.am[n];
            if (p.status) p.status[b] = anybad ? kEData : kOk;
        }
        __syncthreads();
        const int n = s.bi[0], anybad = s.bi[1];
        for (int j = tid; j < R; j += NT) {
            int v = -1;
            if (!anybad) v = j < n ? s.tok[j] : (j == n ? s.am[n] : -1);
            if (SV_IN_SEQ((size_t)b * R + j, (long long)p.B * R, p.status, b)) p.out1[(size_t)b * R + j] = v;
        }
        if (p.probs_dbg) {  // q(x) is 1 iff x is the argmax; greedy drafts have p(x) = 1
            float* dbg = p.probs_dbg;
            for (int j = tid; j < gamma; j += NT) {
                dbg[((size_t)b * gamma + j) * 2 + 0] = (s.tok[j] == s.am[j]) ? 1.f : 0.f;
                dbg[((size_t)b * gamma + j) * 2 + 1] = 1.f;
            }
        }
    } else if (p.mode == kArgSample) {
        int anybad = 0;
        for (int i = 0; i < R; ++i) anybad |= s.bad[i];
        for (int j = tid; j < R; j += NT) p.out0[(size_t)b * R + j] = s.bad[j] ? -1 : s.am[j];
        if (tid == 0 && p.status) p.status[b] = anybad ? kEData : kOk;
    } else {  // tree
        const int N = R;
        for (int i = tid; i < N; i += NT) {
            s.tok[i] = p.node_tokens[base + i];
            s.par[i] = p.parent[base + i];
            s.dep[i] = p.depth[base + i];
        }
        __syncthreads();
        const int W = p.max_depth + 1;
        if (tid == 0) {
            int bad = (s.par[0] != -1) || (s.dep[0] != 0);
            for (int i = 0; i < N; ++i) bad |= s.bad[i];
            for (int i = 1; i < N && !bad; ++i) {
                const int pi = s.par[i];
                if (pi < 0 || pi >= i) {
                    bad = 1;
                    break;
                }
                bad |= (s.dep[i] != s.dep[pi] + 1) || (s.tok[i] < 0) || (s.tok[i] >= p.V) ||
                       (s.dep[i] > p.max_depth);
            }
            int dstar = 0;
            if (!bad) {
                // s.path doubles as the accepted flags: acc[i] = acc[parent] && tok == argmax(parent)
                s.path[0] = 1;
                for (int i = 1; i < N; ++i) {
                    const int pi = s.par[i];
                    s.path[i] = s.path[pi] && (s.tok[i] == s.am[pi]);
                    if (s.path[i] && s.dep[i] > s.dep[dstar]) dstar = i;
                }
            }
            s.bi[0] = bad;
            s.bi[1] = dstar;
            s.bi[2] = bad ? 0 : s.dep[dstar];
            p.out0[b] = bad ? -1 : s.dep[dstar];
            p.out3[b] = bad ? -1 : s.am[dstar];
            if (p.status) p.status[b] = bad ? kEData : kOk;
        }
        __syncthreads();
        const int bad = s.bi[0], dstar = s.bi[1], alen = s.bi[2];
        if (tid == 0 && !bad) {
            for (int node = dstar;; node = s.par[node]) {
                if (!SV_IN_SEQ(node, N, p.status, b) || !SV_IN_SEQ(s.dep[node], kMaxN, p.status, b)) break;
                s.pn[s.dep[node]] = node;
                if (node == 0) break;
            }
        }
        __syncthreads();
        for (int j = tid; j < W; j += NT) {
            int pn = -1, tk = -1;
            if (!bad && j <= alen) pn = s.pn[j];
            if (!bad && j < alen) tk = s.tok[s.pn[j + 1]];
            if (!bad && j == alen) tk = s.am[dstar];
            if (SV_IN_SEQ((size_t)b * W + j, (long long)p.B * W, p.status, b)) {
                p.out1[(size_t)b * W + j] = pn;
                p.out2[(size_t)b * W + j] = tk;
            }
        }
    }
}

template <typename E>
__global__ void __launch_bounds__(NT) argmax_kernel(const __grid_constant__ ArgmaxParams p) {
    __shared__ SharedA s;
    const long long per_b = (long long)p.rows_per_b * p.V;
    const long long total = per_b * p.B;
    const long long e0 = (long long)blockIdx.x * p.chunk;
    const long long e1 = min(total, e0 + (long long)p.chunk);
    if (e0 >= e1) return;
    for (long long e = e0; e < e1;) {
        const long long r = e / p.V;
        const int i0 = (int)(e - r * p.V);
        const int i1 = (int)min((long long)p.V, i0 + (e1 - e));
        segment<E>(p, r, i0, i1);
        e += i1 - i0;
    }
    if ((threadIdx.x & 31) == 0) __threadfence();  // order every warp's atomicMax before the arrivals
    __syncthreads();
    const long long bfirst = e0 / per_b, blast = (e1 - 1) / per_b;
    for (long long b = bfirst; b <= blast; ++b) {
        if (threadIdx.x == 0) {
            const long long lo = max(e0, b * per_b), hi = min(e1, (b + 1) * per_b);
            const unsigned long long n = (unsigned long long)(hi - lo);
            const unsigned long long old = atomicAdd(&p.cnt[b], n);
            const int last = old + n == (unsigned long long)per_b;
            if (last) p.cnt[b] = 0ull;
            s.bi[7] = last;
        }
        __syncthreads();
        if (s.bi[7]) {
            __threadfence();
            resolve(p, s, (int)b);
        }
        __syncthreads();
    }
}

}  // namespace

int argmax_ctas_per_sm(int dtype) {
    static const int f32 = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, argmax_kernel<float>, NT, 0) != cudaSuccess || n < 1) n = 1;
        return n;
    }();
    static const int b16 = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, argmax_kernel<bf16_t>, NT, 0) != cudaSuccess || n < 1) n = 1;
        return n;
    }();
    return dtype == 0 ? f32 : b16;
}

cudaError_t launch_argmax(const ArgmaxParams& p, int dtype, int grid, cudaStream_t stream) {
    if (dtype == 0)
        argmax_kernel<float><<<grid, NT, 0, stream>>>(p);
    else
        argmax_kernel<bf16_t><<<grid, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

SV_DEBUG_READER(argmax)

}  // namespace sv
