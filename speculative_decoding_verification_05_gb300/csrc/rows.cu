// Row-task kernel: modified rejection sampling for temperature > 0.
//
// One thread-block cluster handles one task (b, k): target row k of sequence
// b and, for k < gamma, draft row k. The vocabulary is split across the C
// CTAs of the cluster; each CTA stages its slice of both rows in shared memory
// with bulk asynchronous copies (one HBM pass), and the cluster combines
// partial results through distributed shared memory:
//
//   1. row maxima                       (exchange 1)
//   2. S = sum exp2((z - m) log2e / T)  (exchange 2)
//   3. top-k / top-p thresholds by a cluster-wide radix select on the raw
//      logit keys (one exchange per digit pass)
//   4. acceptance test u < min(1, q(x)/p(x))   ("Accelerating Large Language
//      Model Decoding with Speculative Sampling", "改进的拒绝采样")
//   5. for a rejected row: inverse-CDF draw from max(0, q - p); for the last
//      target row: the bonus draw from q (same section, second bullet). The
//      draw is computed from shared memory, no second HBM pass.
//   6. the last task of sequence b to finish (atomic arrival counter, no
//      waiting) resolves the first rejection and writes the outputs.
//
// The same kernel serves the mentor variant's first stage (records only, no
// resolve) and spec_sample (one row per task, a plain draw).

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kMaxC = 16;
constexpr int kMaxG1 = 256;  // SPEC_MAX_GAMMA + 1

struct alignas(16) Shared {
    uint64_t bar;
    int timeout;
    int mail_tok;          // rank 0: the drawn token (written by the owner CTA)
    float mail_max[3];     // exchange 1 (maxima, timeout flag)
    float mail_sum[2];     // exchange 2
    float mail_w;          // draw: this CTA's total weight
    float mail_aux;        // masked kept mass
    float red[NW][2];
    float all[kMaxC + 1];
    float hist[2][256];    // published radix histograms (double-buffered)
    float htot[256];
    float warp_tot[NW];
    float warp_pre[NW + 1];
    int bi[8];
    float bf[8];
    int rec_flags[kMaxG1];
    int rec_tok[kMaxG1];
};

SV_DEV size_t round128(size_t x) { return (x + 127) & ~size_t(127); }

// Geometry of one CTA's slice [v0, v1) of a row in global memory and its
// 16-byte-aligned copy in shared memory.
struct Geo {
    uintptr_t lo;     // 16-aligned global address of smem vector 0
    uintptr_t a0, a1; // exact byte range of the slice
    uintptr_t b0, b1; // bulk-copied interior (empty if b1 <= b0)
    int nvec;         // 16-byte vectors in the smem buffer
    int first;        // element index of smem element 0 (may precede v0)
};

SV_DEV Geo make_geo(const void* row, int v0, int v1, int es) {
    Geo g;
    g.a0 = (uintptr_t)row + (uintptr_t)v0 * es;
    g.a1 = (uintptr_t)row + (uintptr_t)v1 * es;
    g.lo = g.a0 & ~uintptr_t(15);
    const uintptr_t hi = (g.a1 + 15) & ~uintptr_t(15);
    g.b0 = (g.a0 + 15) & ~uintptr_t(15);
    g.b1 = g.a1 & ~uintptr_t(15);
    g.nvec = (v1 > v0) ? (int)((hi - g.lo) >> 4) : 0;
    g.first = v0 - (int)((g.a0 - g.lo) / es);
    if (g.nvec == 0) g.b1 = g.b0;
    return g;
}

SV_DEV uint32_t bulk_bytes(const Geo& g) { return g.b1 > g.b0 ? (uint32_t)(g.b1 - g.b0) : 0u; }

SV_DEV void issue_bulk(const Geo& g, uint4* buf, uint64_t* bar) {
    const uint32_t total = bulk_bytes(g);
    char* dst = reinterpret_cast<char*>(buf) + (g.b0 - g.lo);
    const char* src = reinterpret_cast<const char*>(g.b0);
    for (uint32_t off = 0; off < total; off += 32768u) {
        const uint32_t n = min(32768u, total - off);
        bulk_g2s(dst + off, src + off, n, bar);
    }
}

// Scalar head/tail of the slice and -inf padding of the smem slots outside it.
template <typename E>
SV_DEV void fill_edges(const Geo& g, uint4* buf) {
    constexpr int es = sizeof(E);
    const int nslots = g.nvec * (16 / es);
    int head, tail_start;
    if (g.b1 > g.b0) {
        head = (int)((g.b0 - g.lo) / es);
        tail_start = (int)((g.b1 - g.lo) / es);
    } else {
        head = nslots;
        tail_start = nslots;
    }
    const int ntail = nslots - tail_start;
    E* e = reinterpret_cast<E*>(buf);
    for (int t = threadIdx.x; t < head + ntail; t += NT) {
        const int slot = t < head ? t : tail_start + (t - head);
        const uintptr_t ga = g.lo + (uintptr_t)slot * es;
        if (ga >= g.a0 && ga < g.a1) {
            e[slot] = *reinterpret_cast<const E*>(ga);
        } else {
            if constexpr (es == 4)
                reinterpret_cast<uint32_t*>(buf)[slot] = VecTraits<float>::kNegInfBits;
            else
                reinterpret_cast<uint16_t*>(buf)[slot] = (uint16_t)VecTraits<bf16_t>::kNegInfBits;
        }
    }
}

// Vectors [j0, j1) of this thread: a contiguous run of K vectors (K odd keeps
// the 16-byte shared loads of a quarter-warp on distinct bank groups).
SV_DEV int per_thread(int nvec) { return ((nvec + NT - 1) / NT) | 1; }

// Block-wide reduction of two floats (op: 0 = max, 1 = sum); result to all threads.
SV_DEV void block_reduce2(Shared& s, float& a, float& b, int op) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (op == 0) {
        a = warp_max(a);
        b = warp_max(b);
    } else {
        a = warp_sum(a);
        b = warp_sum(b);
    }
    if (lane == 0) {
        s.red[warp][0] = a;
        s.red[warp][1] = b;
    }
    __syncthreads();
    float x = s.red[0][0], y = s.red[0][1];
    for (int w = 1; w < NW; ++w) {
        if (op == 0) {
            x = fmaxf(x, s.red[w][0]);
            y = fmaxf(y, s.red[w][1]);
        } else {
            x += s.red[w][0];
            y += s.red[w][1];
        }
    }
    a = x;
    b = y;
    __syncthreads();
}

// Gather mail[0..n) of every CTA of the cluster into out[r * n + i] (local
// smem), after a cluster barrier that publishes the mailboxes.
SV_DEV void cluster_gather(cg::cluster_group& cl, float* mail, float* out, int n, int C) {
    cl.sync();
    for (int t = threadIdx.x; t < C * n; t += NT) {
        const int r = t / n, i = t - r * n;
        out[t] = cl.map_shared_rank(mail, r)[i];
    }
    __syncthreads();
}

// Cluster-wide radix selection: the largest key tau among keys >= floor_key
// whose weight W(key >= tau) reaches `target`; weight 1 (count) or the mass
// exp2(x c2 - mc). If the total weight falls short (rounding), the smallest
// key is chosen. Returns tau's key and W(key >= tau).
template <typename E, bool MASS>
SV_DEV void radix_select(cg::cluster_group& cl, Shared& s, const uint4* buf, int nvec, int C,
                         uint32_t floor_key, float target, float c2, float mc, uint32_t& tau_key,
                         float& w_at) {
    using T = VecTraits<E>;
    constexpr int npass = sizeof(E) == 4 ? 4 : 2;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = per_thread(nvec);
    const int j0 = tid * K, j1 = min(j0 + K, nvec);
    uint32_t prefix = 0;
    float A = 0.f, wsel = 0.f;
    for (int pass = 0; pass < npass; ++pass) {
        const int shift = 24 - 8 * pass;
        float* h = s.hist[pass & 1];
        for (int i = tid; i < 256; i += NT) h[i] = 0.f;
        __syncthreads();
        for (int j = j0; j < j1; ++j) {
            float x[T::kN];
            T::unpack(buf[j], x);
#pragma unroll
            for (int e = 0; e < T::kN; ++e) {
                const uint32_t key = f32_key(x[e]);
                const bool match = key >= floor_key &&
                                   (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8)));
                if (match) atomicAdd(&h[(key >> shift) & 255u], MASS ? ex2(fmaf(x[e], c2, -mc)) : 1.f);
            }
        }
        __syncthreads();
        cl.sync();
        for (int i = tid; i < 256; i += NT) {
            float t = 0.f;
            for (int r = 0; r < C; ++r) t += cl.map_shared_rank(h, r)[i];
            s.htot[i] = t;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l, scanned from the top
            float seg = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) seg += s.htot[255 - 8 * lane - j];
            float total;
            const float pre = warp_seq_exclusive(seg, &total);
            const bool hit = A + (pre + seg) >= target;
            const unsigned hits = __ballot_sync(0xFFFFFFFFu, hit);
            int d = -1;
            float a_new = 0.f, cum = 0.f;
            if (hits) {
                const int f = __ffs(hits) - 1;
                if (lane == f) {
                    float part = 0.f;
                    for (int j = 0; j < 8; ++j) {
                        const int bin = 255 - 8 * lane - j;
                        const float before = part;
                        part += s.htot[bin];
                        if (A + (pre + part) >= target) {
                            d = bin;
                            a_new = A + (pre + before);
                            cum = A + (pre + part);
                            break;
                        }
                    }
                    if (d < 0) {  // rounding between the lane sum and the bin walk
                        int lastpos = -1;
                        float b4 = 0.f, p2 = 0.f;
                        for (int j = 0; j < 8; ++j) {
                            const int bin = 255 - 8 * lane - j;
                            if (s.htot[bin] > 0.f) {
                                lastpos = bin;
                                b4 = p2;
                            }
                            p2 += s.htot[bin];
                        }
                        d = lastpos;
                        a_new = A + (pre + b4);
                        cum = A + (pre + p2);
                    }
                }
                d = __shfl_sync(0xFFFFFFFFu, d, f);
                a_new = __shfl_sync(0xFFFFFFFFu, a_new, f);
                cum = __shfl_sync(0xFFFFFFFFu, cum, f);
            } else {
                // total weight below target: descend into the lowest non-empty bin
                const unsigned nz = __ballot_sync(0xFFFFFFFFu, seg > 0.f);
                const int f = nz ? 31 - __clz(nz) : 31;
                if (lane == f) {
                    float part = 0.f, before_last = 0.f;
                    int lastpos = 255 - 8 * lane - 7;
                    for (int j = 0; j < 8; ++j) {
                        const int bin = 255 - 8 * lane - j;
                        if (s.htot[bin] > 0.f) {
                            lastpos = bin;
                            before_last = part;
                        }
                        part += s.htot[bin];
                    }
                    d = lastpos;
                    a_new = A + (pre + before_last);
                    cum = A + total;
                }
                d = __shfl_sync(0xFFFFFFFFu, d, f);
                a_new = __shfl_sync(0xFFFFFFFFu, a_new, f);
                cum = __shfl_sync(0xFFFFFFFFu, cum, f);
            }
            if (lane == 0) {
                s.bi[0] = d;
                s.bf[0] = a_new;
                s.bf[1] = cum;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)s.bi[0] << shift;
        A = s.bf[0];
        wsel = s.bf[1];
        __syncthreads();
    }
    if (npass == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    tau_key = prefix;
    w_at = wsel;
}

// Per-row normalisation state after the exchanges.
struct RowNorm {
    float m;      // row max
    float mc;     // m * c2
    float S;      // sum over the whole row
    float thr;    // keep z >= thr (-inf: keep all)
    float Sk;     // kept mass (denominator of q)
    bool bad;
};

// Top-k / top-p thresholds of one row (cluster-wide).
template <typename E>
SV_DEV void row_threshold(cg::cluster_group& cl, Shared& s, const RowParams& p, const uint4* buf,
                          int nvec, RowNorm& rn) {
    using T = VecTraits<E>;
    const int tid = threadIdx.x;
    uint32_t floor_key = 0;
    float Sk = rn.S;
    if (p.transform & kXfTopK) {
        uint32_t kkey;
        float cnt;
        radix_select<E, false>(cl, s, buf, nvec, p.C, 0u, (float)p.top_k, p.c2, rn.mc, kkey, cnt);
        floor_key = kkey;
        // kept mass of the top-k set
        const int K = per_thread(nvec);
        const int j0 = tid * K, j1 = min(j0 + K, nvec);
        float acc = 0.f;
        for (int j = j0; j < j1; ++j) {
            float x[T::kN];
            T::unpack(buf[j], x);
#pragma unroll
            for (int e = 0; e < T::kN; ++e)
                if (f32_key(x[e]) >= kkey) acc += ex2(fmaf(x[e], p.c2, -rn.mc));
        }
        float dummy = 0.f;
        block_reduce2(s, acc, dummy, 1);
        if (tid == 0) s.mail_aux = acc;
        cluster_gather(cl, &s.mail_aux, s.all, 1, p.C);
        Sk = 0.f;
        for (int r = 0; r < p.C; ++r) Sk += s.all[r];
        rn.thr = key_to_f32(kkey);
    }
    if (p.transform & kXfTopP) {
        uint32_t pkey;
        float w;
        radix_select<E, true>(cl, s, buf, nvec, p.C, floor_key, p.top_p * Sk, p.c2, rn.mc, pkey, w);
        rn.thr = key_to_f32(pkey);
        Sk = w;
    }
    rn.Sk = Sk;
}

// Element `idx` of a staged slice buffer as fp32.
template <typename E>
SV_DEV float smem_elem(const uint4* buf, int idx) {
    if constexpr (sizeof(E) == 4) {
        return reinterpret_cast<const float*>(buf)[idx];
    } else {
        return __uint_as_float(((uint32_t)reinterpret_cast<const uint16_t*>(buf)[idx]) << 16);
    }
}

SV_DEV float kept_exp(float x, const RowNorm& rn, float c2, bool xf) {
    return (xf && !(x >= rn.thr)) ? 0.f : ex2(fmaf(x, c2, -rn.mc));
}

// Weighted inverse-CDF draw across the cluster: the smallest index i with
// C_i > u W (C the inclusive prefix in index order; if rounding leaves none,
// the last index with positive weight). `thr_w` is this thread's sequential
// sum over its contiguous vectors, `wfun(j, e)` recomputes one weight in the
// same order. Returns the token on rank 0 (others: unspecified); *W_out gets
// the total weight.
template <typename E, typename WF>
SV_DEV int cluster_draw(cg::cluster_group& cl, Shared& s, float thr_w, float u, int nvec,
                        int first, int C, WF wfun, float* W_out) {
    using T = VecTraits<E>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cl.block_rank();
    float wtot;
    const float lane_pre = warp_seq_exclusive(thr_w, &wtot);
    if (lane == 0) s.warp_tot[warp] = wtot;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int w = 0; w < NW; ++w) {
            s.warp_pre[w] = acc;
            acc += s.warp_tot[w];
        }
        s.warp_pre[NW] = acc;
        s.mail_w = acc;
        s.mail_tok = -1;
    }
    __syncthreads();
    cl.sync();
    if (tid == 0) {
        // sequential prefix over ranks, identical in every CTA of the cluster
        for (int r = 0; r < C; ++r) s.all[r] = *cl.map_shared_rank(&s.mail_w, r);
        float W = 0.f;
        for (int r = 0; r < C; ++r) W += s.all[r];
        const float t = u * W;
        int owner = -1;
        float acc = 0.f, owner_pre = 0.f;
        for (int r = 0; r < C; ++r) {
            if (acc <= t && s.all[r] > 0.f) {
                owner = r;
                owner_pre = acc;
            }
            acc += s.all[r];
        }
        s.bi[4] = owner;
        s.bf[5] = W;
        s.bf[6] = t - owner_pre;
    }
    __syncthreads();
    const int owner = s.bi[4];
    *W_out = s.bf[5];
    if (owner == rank) {
        const float tl = s.bf[6];
        // owner warp
        int ow = -1;
        for (int w = 0; w < NW; ++w)
            if (s.warp_pre[w] <= tl && s.warp_tot[w] > 0.f) ow = w;
        if (warp == ow) {
            const float tw = tl - s.warp_pre[ow];
            const bool cand = lane_pre <= tw && thr_w > 0.f;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, cand);
            const int ol = m ? 31 - __clz(m) : -1;
            if (lane == ol) {
                const float tt = tw - lane_pre;
                const int K = per_thread(nvec);
                const int j0 = tid * K, j1 = min(j0 + K, nvec);
                float acc = 0.f;
                int found = -1, lastpos = -1;
                for (int j = j0; j < j1 && found < 0; ++j) {
#pragma unroll
                    for (int e = 0; e < T::kN; ++e) {
                        const float w = wfun(j, e);
                        if (w > 0.f) lastpos = first + j * T::kN + e;
                        acc += w;
                        if (found < 0 && w > 0.f && acc > tt) found = first + j * T::kN + e;
                    }
                }
                *cl.map_shared_rank(&s.mail_tok, 0) = found >= 0 ? found : lastpos;
            }
        }
    }
    cl.sync();
    return s.mail_tok;
}

template <typename E, bool XF>
__global__ void __launch_bounds__(NT) row_kernel(const __grid_constant__ RowParams p) {
    using T = VecTraits<E>;
    constexpr int es = sizeof(E);
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Shared& s = *reinterpret_cast<Shared*>(smem_raw);
    const int C = p.C;
    const int rank = (int)cl.block_rank();
    const int tid = threadIdx.x;
    const int task = blockIdx.x / C;

    int b, k;
    bool has_draft;
    const E* rowT;
    const E* rowD = nullptr;
    if (p.mode == kModeSample) {
        b = task / p.rows_per_b;
        k = task - b * p.rows_per_b;
        has_draft = false;
        rowT = reinterpret_cast<const E*>(p.target) + (size_t)task * p.V;
    } else {
        b = task / (p.gamma + 1);
        k = task - b * (p.gamma + 1);
        has_draft = k < p.gamma;
        rowT = reinterpret_cast<const E*>(p.target) + (size_t)task * p.V;
        if (has_draft)
            rowD = reinterpret_cast<const E*>(p.draft) + ((size_t)b * p.gamma + k) * p.V;
    }

    const size_t rowbytes = round128((size_t)p.L * es + 32);
    uint4* bufT = reinterpret_cast<uint4*>(smem_raw + round128(sizeof(Shared)));
    uint4* bufD = reinterpret_cast<uint4*>(reinterpret_cast<char*>(bufT) + rowbytes);
    const int v0 = min(rank * p.L, p.V), v1 = min(p.V, v0 + p.L);
    const Geo gT = make_geo(rowT, v0, v1, es);
    const Geo gD = has_draft ? make_geo(rowD, v0, v1, es) : Geo{0, 0, 0, 0, 0, 0, 0};

    // ---- stage both slices in shared memory (one HBM pass) ----
    if (tid == 0) {
        mbar_init(&s.bar, 1);
        s.timeout = 0;
    }
    __syncthreads();
    const uint32_t bulk = bulk_bytes(gT) + (has_draft ? bulk_bytes(gD) : 0u);
    if (tid == 0 && bulk) {
        mbar_arrive_expect_tx(&s.bar, bulk);
        issue_bulk(gT, bufT, &s.bar);
        if (has_draft) issue_bulk(gD, bufD, &s.bar);
    }
    fill_edges<E>(gT, bufT);
    if (has_draft) fill_edges<E>(gD, bufD);
    if (bulk && !mbar_wait_bounded(&s.bar, 0, p.wait_limit)) {
        s.timeout = 1;
        mbar_wait_bounded(&s.bar, 0, p.wait_limit);  // drain our own copies before going on
    }
    __syncthreads();

    const int KT = per_thread(gT.nvec), KD = per_thread(gD.nvec);
    const int jT0 = tid * KT, jT1 = min(jT0 + KT, gT.nvec);
    const int jD0 = tid * KD, jD1 = min(jD0 + KD, gD.nvec);

    // ---- 1. row maxima ----
    float mt = -INFINITY, md = -INFINITY;
    for (int j = jT0; j < jT1; ++j) {
        float x[T::kN];
        T::unpack(bufT[j], x);
#pragma unroll
        for (int e = 0; e < T::kN; ++e) mt = fmaxf(mt, x[e]);
    }
    for (int j = jD0; j < jD1; ++j) {
        float x[T::kN];
        T::unpack(bufD[j], x);
#pragma unroll
        for (int e = 0; e < T::kN; ++e) md = fmaxf(md, x[e]);
    }
    block_reduce2(s, mt, md, 0);
    if (tid == 0) {
        s.mail_max[0] = mt;
        s.mail_max[1] = md;
        s.mail_max[2] = s.timeout ? 1.f : 0.f;
    }
    float* gat = reinterpret_cast<float*>(s.htot);  // scratch for gathers (3 * kMaxC floats)
    cluster_gather(cl, s.mail_max, gat, 3, C);
    RowNorm nT, nD;
    nT.m = -INFINITY;
    nD.m = -INFINITY;
    bool timed_out = false;
    for (int r = 0; r < C; ++r) {
        nT.m = fmaxf(nT.m, gat[3 * r]);
        nD.m = fmaxf(nD.m, gat[3 * r + 1]);
        timed_out |= gat[3 * r + 2] != 0.f;
    }
    nT.mc = nT.m * p.c2;
    nD.mc = nD.m * p.c2;
    nT.thr = -INFINITY;
    nD.thr = -INFINITY;
    __syncthreads();

    // ---- 2. sums of exponentials ----
    float sT = 0.f, sD = 0.f;
    for (int j = jT0; j < jT1; ++j) {
        float x[T::kN];
        T::unpack(bufT[j], x);
#pragma unroll
        for (int e = 0; e < T::kN; ++e) sT += ex2(fmaf(x[e], p.c2, -nT.mc));
    }
    for (int j = jD0; j < jD1; ++j) {
        float x[T::kN];
        T::unpack(bufD[j], x);
#pragma unroll
        for (int e = 0; e < T::kN; ++e) sD += ex2(fmaf(x[e], p.c2, -nD.mc));
    }
    const float sT_thr = sT;  // this thread's sequential share, reused for the bonus draw
    block_reduce2(s, sT, sD, 1);
    if (tid == 0) {
        s.mail_sum[0] = sT;
        s.mail_sum[1] = sD;
    }
    cluster_gather(cl, s.mail_sum, gat, 2, C);
    nT.S = 0.f;
    nD.S = 0.f;
    for (int r = 0; r < C; ++r) {
        nT.S += gat[2 * r];
        nD.S += gat[2 * r + 1];
    }
    __syncthreads();
    nT.bad = !(nT.S > 0.f && nT.S <= 3.0e38f);
    nD.bad = has_draft && !(nD.S > 0.f && nD.S <= 3.0e38f);
    nT.Sk = nT.S;
    nD.Sk = nD.S;

    // ---- 3. sampling transforms ----
    if constexpr (XF) {
        // every CTA of the cluster takes the same branches (the flags are cluster-uniform)
        if (!nT.bad) row_threshold<E>(cl, s, p, bufT, gT.nvec, nT);
        if (has_draft && !nD.bad) row_threshold<E>(cl, s, p, bufD, gD.nvec, nD);
    }

    const bool bad_rows = nT.bad || nD.bad || timed_out;

    // ---- 4. acceptance test ----
    if (tid == 0) {
        int acc = 0, tokbad = 0;
        float q = 0.f, pd = 0.f;
        if (has_draft && !bad_rows) {
            const int x = p.draft_tokens[(size_t)b * p.gamma + k];
            if (x < 0 || x >= p.V) {
                tokbad = 1;
            } else {
                const float zt = T::load1(rowT + x), zd = T::load1(rowD + x);
                q = kept_exp(zt, nT, p.c2, XF) / nT.Sk;
                pd = kept_exp(zd, nD, p.c2, XF) / nD.Sk;
                const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
                const float ratio = pd > 0.f ? q / pd : (q > 0.f ? INFINITY : 0.f);
                acc = u < ratio;
            }
        }
        s.bi[1] = acc;
        s.bi[2] = tokbad;
        s.bf[2] = q;
        s.bf[3] = pd;
    }
    __syncthreads();
    const bool accept = s.bi[1] != 0;
    const bool tokbad = s.bi[2] != 0;
    const bool bad = bad_rows || tokbad;

    // ---- 5. draw (rejected row: max(0, q-p); last row / sample: q) ----
    int token = -1;
    const bool draw = !bad && (p.mode == kModeSample || !has_draft || !accept);
    if (draw) {
        uint32_t pos, purpose;
        if (p.mode == kModeSample) {
            pos = p.pos0 + (uint32_t)k;
            purpose = p.purpose;
        } else {
            pos = (uint32_t)k;
            purpose = kPurposeResample;
        }
        const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, pos, purpose);
        auto wq = [&](int j, int e) -> float {
            float x[T::kN];
            T::unpack(bufT[j], x);
            return kept_exp(x[e], nT, p.c2, XF);
        };
        bool use_q = !has_draft;
        float W = 0.f;
        if (has_draft) {
            const float iT = 1.f / nT.Sk, iD = 1.f / nD.Sk;
            // The two rows' slices start at the same 16-byte phase unless
            // V * sizeof(E) is not a multiple of 16; then the draft element
            // paired with target element i is read by index.
            const bool same_phase = gT.first == gD.first;
            auto wr = [&](int j, int e) -> float {
                float xt[T::kN];
                T::unpack(bufT[j], xt);
                float xd_e;
                if (same_phase) {
                    float xd[T::kN];
                    T::unpack(bufD[j], xd);
                    xd_e = xd[e];
                } else {
                    const int i = gT.first + j * T::kN + e;
                    xd_e = (i >= v0 && i < v1) ? smem_elem<E>(bufD, i - gD.first) : -INFINITY;
                }
                const float qi = kept_exp(xt[e], nT, p.c2, XF) * iT;
                const float pi = kept_exp(xd_e, nD, p.c2, XF) * iD;
                return fmaxf(0.f, qi - pi);
            };
            float tw = 0.f;
            for (int j = jT0; j < jT1; ++j)
#pragma unroll
                for (int e = 0; e < T::kN; ++e) tw += wr(j, e);
            token = cluster_draw<E>(cl, s, tw, u2, gT.nvec, gT.first, C, wr, &W);
            if (!(W > 0.f)) use_q = true;  // (q-p)+ vanished: draw from q
        }
        if (use_q) {
            float tw = 0.f;
            if (XF || has_draft) {
                for (int j = jT0; j < jT1; ++j)
#pragma unroll
                    for (int e = 0; e < T::kN; ++e) tw += wq(j, e);
            } else {
                tw = sT_thr;
            }
            token = cluster_draw<E>(cl, s, tw, u2, gT.nvec, gT.first, C, wq, &W);
        }
    }

    // ---- 6. record, arrival, resolve ----
    if (rank == 0 && tid == 0) {
        const int flags = (accept ? kRecAccept : 0) | (bad ? kRecEData : 0) |
                          (timed_out ? kRecTimeout : 0);
        if (p.mode == kModeSample) {
            p.sample_out[task] = bad ? -1 : token;
            if (bad && p.status) atomicMax(&p.status[b], timed_out ? kETimeout : kEData);
            s.bi[3] = 0;
        } else {
            TaskRec r;
            r.flags = flags;
            r.token = token;
            r.q_x = s.bf[2];
            r.p_x = s.bf[3];
            r.m_t = nT.m;
            r.s_t = nT.Sk;
            r.m_d = nD.m;
            r.s_d = nD.Sk;
            p.recs[task] = r;
            if (has_draft && p.probs_dbg) {
                p.probs_dbg[((size_t)b * p.gamma + k) * 2 + 0] = s.bf[2];
                p.probs_dbg[((size_t)b * p.gamma + k) * 2 + 1] = s.bf[3];
            }
            int last = 0;
            if (p.mode == kModeVerify) {
                __threadfence();
                const unsigned old = atomicAdd(&p.cnt[b], 1u);
                last = old == (unsigned)p.gamma;
                if (last) p.cnt[b] = 0u;
            }
            s.bi[3] = last;
        }
    }
    cl.sync();  // no DSMEM access to this CTA after this point
    if (rank != 0 || s.bi[3] == 0) return;

    // Last arrival for sequence b: resolve the first rejection.
    __threadfence();
    const int G1 = p.gamma + 1;
    for (int i = tid; i < G1; i += NT) {
        const TaskRec* r = p.recs + (size_t)b * G1 + i;
        s.rec_flags[i] = __ldcg(&r->flags);
        s.rec_tok[i] = __ldcg(&r->token);
    }
    __syncthreads();
    if (tid == 0) {
        int n = p.gamma, flags = 0;
        for (int i = 0; i < G1; ++i) flags |= s.rec_flags[i];
        for (int i = 0; i < p.gamma; ++i)
            if (!(s.rec_flags[i] & kRecAccept)) {
                n = i;
                break;
            }
        const int st = (flags & kRecEData) ? kEData : ((flags & kRecTimeout) ? kETimeout : kOk);
        p.accepted[b] = st ? -1 : n;
        p.next_token[b] = st ? -1 : s.rec_tok[n];
        if (p.status) p.status[b] = st;
        s.bi[5] = n;
        s.bi[6] = st;
    }
    __syncthreads();
    const int n = s.bi[5], st = s.bi[6];
    for (int j = tid; j < G1; j += NT) {
        int v = -1;
        if (!st) v = j < n ? p.draft_tokens[(size_t)b * p.gamma + j] : (j == n ? s.rec_tok[n] : -1);
        p.tokens[(size_t)b * G1 + j] = v;
    }
}

template <typename E, bool XF>
cudaError_t launch_t(const RowParams& p, int num_tasks, size_t smem, cudaStream_t stream) {
    auto kern = row_kernel<E, XF>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (p.C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_tasks * p.C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t rows_smem_bytes(int dtype, int L, bool two_rows) {
    const size_t es = dtype == 0 ? 4 : 2;
    const size_t hdr = (sizeof(Shared) + 127) & ~size_t(127);
    const size_t row = ((size_t)L * es + 32 + 127) & ~size_t(127);
    return hdr + (two_rows ? 2 : 1) * row;
}

cudaError_t launch_rows(const RowParams& p, int dtype, int num_tasks, size_t smem,
                        cudaStream_t stream) {
    const bool xf = p.transform != 0;
    if (dtype == 0)
        return xf ? launch_t<float, true>(p, num_tasks, smem, stream)
                  : launch_t<float, false>(p, num_tasks, smem, stream);
    return xf ? launch_t<bf16_t, true>(p, num_tasks, smem, stream)
              : launch_t<bf16_t, false>(p, num_tasks, smem, stream);
}

}  // namespace sv
