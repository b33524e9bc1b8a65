// Mentor (lossy) verification, second stage.
//
// "推测解码的一种最优有损变体", section "解决优化问题": the KL-bounded optimum
// has r_i = min(1, q_i/(alpha p_i)) and s_i ~ max(0, q_i/beta - p_i), with KL
// falling as alpha grows, so alpha is found by bisection; the page lists the
// savings used here: a position whose uniform passes the standard test
// u < min(1, q/p) is accepted without solving, a row with KL(q || p) <= D is
// accepted directly, and the six running sums over the indices sorted by
// rho = q/p are computed once per solved row:
//   cq = sum_{i<=j} q, cp = sum_{i<=j} p, sq = sum_{i>=j} q, sp = sum_{i>=j} p,
//   cl = sum_{i<=j} q ln(q/p), g = (p_j/q_j) sq_j - sp_j.
// For alpha: k = #{rho < alpha}, R = cp_{k-1} - cq_{k-1}/alpha, m = first j
// with g_j <= R, beta = sq_m/(R + sp_m) and
//   KL(alpha) = ln(alpha) cq_{k-1} + (cl_{m-1} - cl_{k-1}) + ln(beta) sq_m.
//
// The row kernel has already written every row's record (maximum, sum, the
// draft token's logit). Each position's outcome depends only on its own rows
// and its own uniforms, so the position kernel (1024 threads, one persistent
// CTA per SM) solves (sequence, position) jobs independently, skipping a job
// once an earlier position of its sequence is known to be rejected; the
// resolve kernel then finds each sequence's first rejection and makes its one
// draw. The sort is a stable LSD radix sort (four 8-bit digit passes) of the
// fp32 keys of ln(rho) in global scratch. The bisection's result (the smallest
// dyadic alpha = j 2^-iters with KL(alpha) <= D) is found by a multiway
// search: each round evaluates KL at up to 1023 interior grid points of the
// current interval in parallel, ten bisection steps at a time. Rejections with
// alpha = 1 (beta = 1) and the bonus token use the verification path's own
// draw, so D = 0 reproduces spec_verify bit for bit.

#include "common.cuh"
#include "draw.cuh"

namespace sv {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int kIPT = 8;          // items per thread per sort tile
constexpr int kTile = NT * kIPT; // 8192
constexpr int kCoarse = 32;      // coarse index stride

struct SharedM {
    uint32_t wcnt[NW][256];      // per-warp digit counts, then offsets
    uint32_t stk[kTile];         // one tile in digit order (keys, indices)
    uint32_t sti[kTile];
    uint32_t hist[4][256];       // all four digit histograms
    uint32_t base[256];          // next free global position per bucket
    uint32_t dtot[256];          // tile: per-digit count, start, global offset
    uint32_t dstart[256];
    uint32_t gofs[256];
    double dred[NW];
    float wsum[5][NW];           // solve: per-warp chunk totals
    float woff[5][NW];           //        and chunk offsets
    int ibuf[NW];
    int bi[8];
    double bd[8];
    DrawShared draw;
};

SV_DEV double block_sum_d(SharedM& s, double v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) s.dred[warp] = v;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < NW; ++w) t += s.dred[w];
    __syncthreads();
    return t;
}

template <typename E>
struct Row {
    const E* rt;       // target / draft rows
    const E* rd;
    float mtc, mdc;    // m * c2
    float c2, inv_t;
    float iSt, iSd;    // 1 / S
    float lnr0;        // -(m_t - m_d)/T - ln S_t + ln S_d
};

template <typename E>
SV_DEV void qpl(const Row<E>& r, int i, float& q, float& p, float& l) {
    const float zt = VecTraits<E>::load1(r.rt + i), zd = VecTraits<E>::load1(r.rd + i);
    q = ex2(fmaf(zt, r.c2, -r.mtc)) * r.iSt;
    p = ex2(fmaf(zd, r.c2, -r.mdc)) * r.iSd;
    l = (zt - zd) * r.inv_t + r.lnr0;
}

// Stable LSD radix sort of (key, idx) pairs, ascending, four 8-bit digits.
// k0/i0 hold the input; the sorted result ends in k0/i0 again. A key's digits
// do not change from pass to pass, so one read of the keys builds all four
// digit histograms. Each tile of kTile items is ranked per warp (stable),
// laid out in digit order in shared memory, and written out from there so
// that consecutive threads write consecutive positions of a bucket.
SV_DEV void radix_sort(SharedM& s, uint32_t* k0, uint32_t* i0, uint32_t* k1, uint32_t* i1, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    for (int e = tid; e < 4 * 256; e += NT) (&s.hist[0][0])[e] = 0u;
    __syncthreads();
    for (int ib = tid; ib < n; ib += NT * 8) {  // eight loads in flight per thread
        uint32_t kk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) kk[u] = ib + u * NT < n ? __ldcg(k0 + ib + u * NT) : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (ib + u * NT < n) {
#pragma unroll
                for (int g = 0; g < 4; ++g) atomicAdd(&s.hist[g][(kk[u] >> (8 * g)) & 255u], 1u);
            }
        }
    }
    __syncthreads();
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 8 * pass;
        uint32_t* sk = pass & 1 ? k1 : k0;
        uint32_t* si = pass & 1 ? i1 : i0;
        uint32_t* dk = pass & 1 ? k0 : k1;
        uint32_t* di = pass & 1 ? i0 : i1;
        // exclusive bucket starts of this digit
        if (warp == 0) {
            uint32_t c[8], seg = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = s.hist[pass][lane * 8 + j];
                seg += c[j];
            }
            uint32_t incl = seg;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            uint32_t run = incl - seg;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s.base[lane * 8 + j] = run;
                run += c[j];
            }
        }
        __syncthreads();
        for (int t0 = 0; t0 < n; t0 += kTile) {
            for (int e = tid; e < NW * 256; e += NT) (&s.wcnt[0][0])[e] = 0u;
            // warp w owns items [w*256, w*256+256) of the tile
            uint32_t key[kIPT], idv[kIPT], rank[kIPT];
            int dig[kIPT];
#pragma unroll
            for (int r = 0; r < kIPT; ++r) {
                const int i = t0 + warp * (32 * kIPT) + r * 32 + lane;
                const bool ok = i < n;
                key[r] = ok ? __ldcg(sk + i) : 0u;
                idv[r] = ok ? __ldcg(si + i) : 0u;
                dig[r] = ok ? (int)((key[r] >> shift) & 255u) : -1;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kIPT; ++r) {
                const bool ok = dig[r] >= 0;
                const unsigned act = __ballot_sync(0xFFFFFFFFu, ok);
                unsigned peers = __match_any_sync(0xFFFFFFFFu, dig[r]);
                peers &= act;
                const int leader = peers ? __ffs(peers) - 1 : lane;
                uint32_t old = 0;
                if (ok && lane == leader) {
                    old = s.wcnt[warp][dig[r]];
                    s.wcnt[warp][dig[r]] = old + __popc(peers);
                }
                old = __shfl_sync(0xFFFFFFFFu, old, leader);
                rank[r] = old + __popc(peers & lt);
                __syncwarp();
            }
            __syncthreads();
            // tile-local starts: digit-major, warps in order inside a digit
            const int d = tid >> 2, q = tid & 3;
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = s.wcnt[q * 8 + j][d];
                sum += c[j];
            }
            uint32_t incl = sum;
            const uint32_t v1 = __shfl_up_sync(0xFFFFFFFFu, incl, 1, 4);
            if (q >= 1) incl += v1;
            const uint32_t v2 = __shfl_up_sync(0xFFFFFFFFu, incl, 2, 4);
            if (q >= 2) incl += v2;
            if (q == 3) s.dtot[d] = incl;
            __syncthreads();
            if (warp == 0) {
                uint32_t cc[8], seg = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    cc[j] = s.dtot[lane * 8 + j];
                    seg += cc[j];
                }
                uint32_t in2 = seg;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, in2, o);
                    if (lane >= o) in2 += v;
                }
                uint32_t run = in2 - seg;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int dd = lane * 8 + j;
                    s.dstart[dd] = run;
                    s.gofs[dd] = s.base[dd] - run;  // global position = gofs + tile-local position
                    s.base[dd] += cc[j];
                    run += cc[j];
                }
            }
            __syncthreads();
            {
                uint32_t run = s.dstart[d] + incl - sum;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    s.wcnt[q * 8 + j][d] = run;
                    run += c[j];
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kIPT; ++r) {
                if (dig[r] >= 0) {
                    const uint32_t lp = s.wcnt[warp][dig[r]] + rank[r];
                    s.stk[lp] = key[r];
                    s.sti[lp] = idv[r];
                }
            }
            __syncthreads();
            const int cnt = min(kTile, n - t0);
            for (int lp = tid; lp < cnt; lp += NT) {
                const uint32_t kv = s.stk[lp];
                const uint32_t pos = s.gofs[(kv >> shift) & 255u] + (uint32_t)lp;
                dk[pos] = kv;
                di[pos] = s.sti[lp];
            }
            __syncthreads();
        }
        __threadfence_block();
        __syncthreads();
    }
}

// Evaluate KL(alpha) and beta from the sorted arrays (global scratch).
struct Arrays {
    const float* L;   // sorted ln rho
    const float* CQ;  // inclusive prefix of q
    const float* CP;
    const float* CL;  // inclusive prefix of q ln rho
    const float* SQ;  // inclusive suffix of q
    const float* SP;
    const float* G;   // sq_j / rho_j - sp_j
    const float* cL;  // coarse copies (shared memory): every kCoarse-th entry
    const float* cG;
    int n, nc;
};

SV_DEV int count_less(const Arrays& a, double lnalpha) {
    // number of j with L[j] < lnalpha (L ascending): coarse search in smem, then fine
    int lo = 0, hi = a.nc;  // first coarse block whose head is >= lnalpha
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((double)a.cL[mid] < lnalpha) lo = mid + 1; else hi = mid;
    }
    int flo = max(0, (lo - 1) * kCoarse), fhi = min(a.n, lo * kCoarse);
    while (flo < fhi) {
        const int mid = (flo + fhi) >> 1;
        if ((double)__ldcg(a.L + mid) < lnalpha) flo = mid + 1; else fhi = mid;
    }
    return flo;
}

SV_DEV int first_g_le(const Arrays& a, double R) {
    // first j with G[j] <= R (G non-increasing)
    int lo = 0, hi = a.nc;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((double)a.cG[mid] <= R) hi = mid; else lo = mid + 1;
    }
    int flo = max(0, (lo - 1) * kCoarse), fhi = min(a.n, lo * kCoarse);
    if (lo == a.nc) fhi = a.n;
    while (flo < fhi) {
        const int mid = (flo + fhi) >> 1;
        if ((double)__ldcg(a.G + mid) <= R) fhi = mid; else flo = mid + 1;
    }
    return flo;
}

SV_DEV double kl_at(const Arrays& a, double alpha, double* beta_out) {
    const double lna = (double)logf((float)alpha);  // fp32 log: ~1e-7, far inside the KL tolerance
    const int k = count_less(a, lna);
    const double qlow = k ? (double)__ldcg(a.CQ + k - 1) : 0.0;
    const double plow = k ? (double)__ldcg(a.CP + k - 1) : 0.0;
    const double llow = k ? (double)__ldcg(a.CL + k - 1) : 0.0;
    const double R = plow - qlow / alpha;
    int m = max(first_g_le(a, R), k);
    m = min(m, a.n - 1);
    const double sqm = (double)__ldcg(a.SQ + m), spm = (double)__ldcg(a.SP + m);
    const double beta = sqm / (R + spm);
    const double lmid = (m ? (double)__ldcg(a.CL + m - 1) : 0.0) - llow;
    if (beta_out) *beta_out = beta;
    return lna * qlow + lmid + (double)logf((float)beta) * sqm;
}

// Solves one row pair: alpha (the bisection result) and beta. kl0 > D > 0.
template <typename E>
SV_DEV void solve(SharedM& s, float* coarse, const MentorParams& p, const Row<E>& r, uint32_t* k0,
                  uint32_t* i0, uint32_t* k1, uint32_t* i1, float* A, double* alpha_out, float* beta_out) {
    const int tid = threadIdx.x;
    const int V = p.V;
    const int nc = (V + kCoarse - 1) / kCoarse;
    radix_sort(s, k0, i0, k1, i1, V);
    // sorted arrays: L, CQ, CP, CL (prefix), SQ, SP (suffix), G
    float* L = A;
    float* CQ = A + V;
    float* CP = A + 2 * (size_t)V;
    float* CL = A + 3 * (size_t)V;
    float* SQ = A + 4 * (size_t)V;
    float* SP = A + 5 * (size_t)V;
    float* Gg = A + 6 * (size_t)V;
    // q, p and ln rho per index were left in CQ, CP, CL by the KL pass. Warp w
    // owns the contiguous chunk [w cw, (w + 1) cw) of sorted positions and
    // walks it 32 positions at a time, so every pass below is coalesced.
    const int lane = tid & 31, warp = tid >> 5;
    const int cw = ((V + NW - 1) / NW + 31) & ~31;
    const int w0 = min(V, warp * cw), w1 = min(V, w0 + cw);
    // gather into sorted order: L, and q, p in the SQ, SP slots
    for (int jb = w0; jb < w1; jb += 4 * 32) {
        int idx[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = jb + u * 32 + lane;
            idx[u] = j < w1 ? (int)__ldcg(i0 + j) : -1;
        }
        float lv[4], qv[4], pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (idx[u] >= 0) {
                lv[u] = __ldcg(CL + idx[u]);
                qv[u] = __ldcg(CQ + idx[u]);
                pv[u] = __ldcg(CP + idx[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (idx[u] >= 0) {
                const int j = jb + u * 32 + lane;
                L[j] = lv[u];
                SQ[j] = qv[u];
                SP[j] = pv[u];
            }
        }
    }
    __syncthreads();
    // chunk-local prefix sums (q, p, q ln rho) and suffix sums (q, p): a warp
    // scan per 32 positions plus a running carry
    {
        float cq = 0.f, cp = 0.f, cl = 0.f;
        for (int jb = w0; jb < w1; jb += 32) {
            const int j = jb + lane;
            const bool ok = j < w1;
            float q = ok ? __ldcg(SQ + j) : 0.f, pp = ok ? __ldcg(SP + j) : 0.f;
            float ql = ok ? q * __ldcg(L + j) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a1 = __shfl_up_sync(0xFFFFFFFFu, q, o), a2 = __shfl_up_sync(0xFFFFFFFFu, pp, o),
                            a3 = __shfl_up_sync(0xFFFFFFFFu, ql, o);
                if (lane >= o) {
                    q += a1;
                    pp += a2;
                    ql += a3;
                }
            }
            if (ok) {
                CQ[j] = cq + q;
                CP[j] = cp + pp;
                CL[j] = cl + ql;
            }
            cq += __shfl_sync(0xFFFFFFFFu, q, 31);
            cp += __shfl_sync(0xFFFFFFFFu, pp, 31);
            cl += __shfl_sync(0xFFFFFFFFu, ql, 31);
        }
        float sq = 0.f, sp = 0.f;
        for (int jb = w0 + ((w1 - w0 - 1) & ~31); w1 > w0 && jb >= w0; jb -= 32) {
            const int j = jb + lane;
            const bool ok = j < w1;
            float q = ok ? __ldcg(SQ + j) : 0.f, pp = ok ? __ldcg(SP + j) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a1 = __shfl_down_sync(0xFFFFFFFFu, q, o), a2 = __shfl_down_sync(0xFFFFFFFFu, pp, o);
                if (lane + o < 32) {
                    q += a1;
                    pp += a2;
                }
            }
            if (ok) {
                SQ[j] = sq + q;
                SP[j] = sp + pp;
            }
            sq += __shfl_sync(0xFFFFFFFFu, q, 0);
            sp += __shfl_sync(0xFFFFFFFFu, pp, 0);
        }
        if (lane == 0) {
            s.wsum[0][warp] = cq;
            s.wsum[1][warp] = cp;
            s.wsum[2][warp] = cl;
            s.wsum[3][warp] = sq;
            s.wsum[4][warp] = sp;
        }
    }
    __syncthreads();
    // chunk offsets in a fixed order: prefixes left to right, suffixes right to left
    if (tid < 5) {
        float acc = 0.f;
        if (tid < 3) {
            for (int w = 0; w < NW; ++w) {
                s.woff[tid][w] = acc;
                acc += s.wsum[tid][w];
            }
        } else {
            for (int w = NW - 1; w >= 0; --w) {
                s.woff[tid][w] = acc;
                acc += s.wsum[tid][w];
            }
        }
    }
    __syncthreads();
    {
        const float oq = s.woff[0][warp], op = s.woff[1][warp], ol = s.woff[2][warp];
        const float xq = s.woff[3][warp], xp = s.woff[4][warp];
        for (int j = w0 + lane; j < w1; j += 32) {
            CQ[j] = oq + __ldcg(CQ + j);
            CP[j] = op + __ldcg(CP + j);
            CL[j] = ol + __ldcg(CL + j);
            const float sqj = xq + __ldcg(SQ + j), spj = xp + __ldcg(SP + j);
            SQ[j] = sqj;
            SP[j] = spj;
            Gg[j] = sqj * ex2(-__ldcg(L + j) * 1.4426950408889634f) - spj;
        }
    }
    __threadfence_block();
    __syncthreads();
    for (int c = tid; c < nc; c += NT) {
        coarse[c] = __ldcg(L + c * kCoarse);
        coarse[nc + c] = __ldcg(Gg + c * kCoarse);
    }
    __syncthreads();
    Arrays ar{L, CQ, CP, CL, SQ, SP, Gg, coarse, coarse + nc, V, nc};
    // multiway search for the smallest grid alpha with KL(alpha) <= D
    double lo = 0.0, hi = 1.0;
    int left = p.iters;
    while (left > 0) {
        const int bits = min(10, left);
        const int npts = (1 << bits) - 1;
        const double step = (hi - lo) / (double)(1 << bits);
        int feas = 0;
        if (tid < npts) {
            const double a = lo + (double)(tid + 1) * step;
            feas = kl_at(ar, a, nullptr) <= (double)p.kl_bound;
        }
        // smallest feasible interior point (monotone KL): first set bit
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, feas);
        if ((tid & 31) == 0) s.ibuf[tid >> 5] = bal ? (tid + __ffs(bal) - 1) : 0x7FFFFFFF;
        __syncthreads();
        if (tid == 0) {
            int f = 0x7FFFFFFF;
            for (int w = 0; w < NW; ++w) f = min(f, s.ibuf[w]);
            s.bi[2] = f;
        }
        __syncthreads();
        const int f = s.bi[2];
        __syncthreads();
        if (f == 0x7FFFFFFF) {
            lo = hi - step;  // only the upper end is feasible
        } else {
            hi = lo + (double)(f + 1) * step;
            lo = hi - step;
        }
        left -= bits;
    }
    *alpha_out = hi;
    if (hi == 1.0) {
        *beta_out = 1.f;
    } else {
        if (tid == 0) {
            double bt;
            kl_at(ar, hi, &bt);
            s.bd[0] = bt;
        }
        __syncthreads();
        *beta_out = (float)s.bd[0];
        __syncthreads();
    }
}

// Position states left for the resolve kernel.
constexpr int kPosAccepted = 1;
constexpr int kPosRejected = 0;        // rejected by the standard test (alpha = 1, beta = 1)
constexpr int kPosRejectedScaled = 2;  // rejected with alpha < 1: resample from max(0, q/beta - p)

// One job per (sequence, position), position-major, so every sequence's first
// position is taken before any second one. Each position's outcome depends
// only on its own rows and its own uniforms, so positions are solved
// independently; a job whose sequence already has an earlier rejection on
// record is skipped (its outcome cannot matter). Positions up to the first
// rejection are never skipped.
template <typename E>
__global__ void __launch_bounds__(NT, 1) mentor_kernel(const __grid_constant__ MentorParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SharedM& s = *reinterpret_cast<SharedM*>(smem_raw);
    float* coarse = reinterpret_cast<float*>(smem_raw + ((sizeof(SharedM) + 15) & ~size_t(15)));
    const int tid = threadIdx.x;
    const int V = p.V, G = p.gamma, G1 = G + 1, R = 2 * G + 1;
    const float c2 = p.c2;
    const size_t slot = blockIdx.x;
    uint32_t* k0 = p.keys + slot * 2 * (size_t)V;
    uint32_t* k1 = k0 + V;
    uint32_t* i0 = p.idx + slot * 2 * (size_t)V;
    uint32_t* i1 = i0 + V;
    float* A = p.arr + slot * 7 * (size_t)V;
    const E* tgt = reinterpret_cast<const E*>(p.target);
    const E* dft = reinterpret_cast<const E*>(p.draft);
    const long long jobs = (long long)p.B * G;

    for (;;) {
        if (tid == 0) s.bi[4] = (int)atomicAdd(p.work, 1u);
        __syncthreads();
        const long long job = s.bi[4];
        if (job >= jobs) break;
        const int k = (int)(job / p.B), b = (int)(job % p.B);
        const size_t pos = (size_t)b * G + k;
        const RowRec* rb = p.rows + (size_t)b * R;
        const RowRec t = load_rec(rb + k), d = load_rec(rb + G1 + k);
        const float q = KeptExp{t.thr, c2, t.m * c2, 1.f}(t.zx) / t.Sk;
        const float pd = KeptExp{d.thr, c2, d.m * c2, 1.f}(d.zx) / d.Sk;
        if (p.probs_dbg && tid == 0) {
            p.probs_dbg[pos * 2 + 0] = q;
            p.probs_dbg[pos * 2 + 1] = pd;
        }
        int fl = 0;
        for (int i = tid; i < R; i += NT) fl |= __ldcg(&rb[i].flags);
        const bool bad = __syncthreads_or(fl & kRecEData) != 0;
        if (tid == 0) s.bi[5] = G - (int)__ldcg(p.rejmark + b) < k;
        __syncthreads();
        const bool skip = s.bi[5] != 0;
        __syncthreads();
        if (bad || skip) continue;

        // the verification path's probabilities and standard test
        const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
        float alpha = -1.f, beta = 0.f;
        int state = accept_test(u, q, pd) ? kPosAccepted : kPosRejected;
        if (state != kPosAccepted) {
            Row<E> r;
            r.rt = tgt + ((size_t)b * G1 + k) * V;
            r.rd = dft + ((size_t)b * G + k) * V;
            r.c2 = c2;
            r.inv_t = p.inv_t;
            r.mtc = t.m * c2;
            r.mdc = d.m * c2;
            r.iSt = 1.f / t.S;
            r.iSd = 1.f / d.S;
            r.lnr0 = -(t.m - d.m) * p.inv_t - logf(t.S) + logf(d.S);
            // KL(q || p), the sort keys, and q, p, ln rho per index for the solve
            float acc_kl = 0.f;
            for (int i = tid; i < V; i += NT) {
                float qq, pp, l;
                qpl(r, i, qq, pp, l);
                acc_kl += qq * l;
                k0[i] = f32_key(l);
                i0[i] = (uint32_t)i;
                A[V + i] = qq;
                A[2 * (size_t)V + i] = pp;
                A[3 * (size_t)V + i] = l;
            }
            const double kl0 = block_sum_d(s, (double)acc_kl);
            if (kl0 <= (double)p.kl_bound) {
                state = kPosAccepted;
                alpha = 0.f;
            } else {
                double a = 1.0;
                beta = 1.f;
                if (p.kl_bound > 0.f) {
                    __threadfence_block();
                    __syncthreads();
                    solve<E>(s, coarse, p, r, k0, i0, k1, i1, A, &a, &beta);
                }
                alpha = (float)a;
                // alpha = 1 is the standard test, which failed
                if (a < 1.0) {
                    const double rho = pd > 0.f ? (double)q / (double)pd : (q > 0.f ? HUGE_VAL : 0.0);
                    state = (double)u < fmin(1.0, rho / a) ? kPosAccepted : kPosRejectedScaled;
                }
            }
        }
        if (tid == 0) {
            if (p.alpha_out) p.alpha_out[pos] = alpha;
            if (p.beta_out) p.beta_out[pos] = beta;
            p.pos_beta[pos] = beta;
            p.pos_state[pos] = state;
            if (state != kPosAccepted) atomicMax(p.rejmark + b, (unsigned)(G - k));
        }
        __syncthreads();
    }
}

// One sequence per CTA pass: n = the first rejected position (gamma if none),
// the one draw at n (resample or bonus), and the outputs. Every position up
// to n was solved by the position kernel.
template <typename E>
__global__ void __launch_bounds__(kDrawNT) mentor_resolve_kernel(const __grid_constant__ MentorParams p) {
    __shared__ DrawShared ds;
    __shared__ int sh[2];
    const int tid = threadIdx.x;
    const int V = p.V, G = p.gamma, G1 = G + 1, R = 2 * G + 1;
    const float c2 = p.c2;
    const E* tgt = reinterpret_cast<const E*>(p.target);
    const E* dft = reinterpret_cast<const E*>(p.draft);
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        const RowRec* rb = p.rows + (size_t)b * R;
        int fl = 0;
        for (int i = tid; i < R; i += kDrawNT) fl |= __ldcg(&rb[i].flags);
        const bool bad = __syncthreads_or(fl & kRecEData) != 0;
        if (tid == 0) {
            int n = G, st = kPosAccepted;
            for (int k = 0; k < G && !bad; ++k) {
                st = __ldcg(p.pos_state + (size_t)b * G + k);
                if (st != kPosAccepted) {
                    n = k;
                    break;
                }
            }
            sh[0] = n;
            sh[1] = st;
        }
        __syncthreads();
        const int n = sh[0], st = sh[1];
        int tok = -1;
        if (!bad) {
            const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)n, kPurposeResample);
            const RowRec t = load_rec(rb + n);
            const E* rt = tgt + ((size_t)b * G1 + n) * V;
            if (n == G) {
                tok = draw_q<E, draw_vec<E>()>(ds, rt, V, t, c2, u2);
            } else {
                const RowRec d = load_rec(rb + G1 + n);
                const E* rd = dft + ((size_t)b * G + n) * V;
                if (st == kPosRejected) {
                    tok = draw_residual<E, draw_vec<E>()>(ds, rt, rd, V, t, d, c2, u2);
                } else {
                    const float beta = __ldcg(p.pos_beta + (size_t)b * G + n);
                    const ResidualW w{KeptExp{t.thr, c2, t.m * c2, (1.f / t.S) * (1.f / beta)},
                                      KeptExp{d.thr, c2, d.m * c2, 1.f / d.S}};
                    float W;
                    tok = block_draw<E, ResidualW, draw_vec<E>()>(ds, rt, rd, V, u2, w, &W);
                    if (!(W > 0.f)) tok = draw_q<E, draw_vec<E>()>(ds, rt, V, t, c2, u2);
                }
            }
        }
        if (tid == 0) {
            p.accepted[b] = bad ? -1 : n;
            p.next_token[b] = bad ? -1 : tok;
            if (p.status) p.status[b] = bad ? kEData : kOk;
        }
        for (int j = tid; j <= G; j += kDrawNT) {
            int v = -1;
            if (!bad) v = j < n ? __ldcg(&rb[j].x) : (j == n ? tok : -1);
            p.tokens[(size_t)b * G1 + j] = v;
        }
        for (int k = tid; k < G; k += kDrawNT) {
            if (bad || k > n) {
                if (p.alpha_out) p.alpha_out[(size_t)b * G + k] = NAN;
                if (p.beta_out) p.beta_out[(size_t)b * G + k] = NAN;
            }
        }
        __syncthreads();
    }
}

}  // namespace

size_t mentor_smem_bytes(int V) {
    const int nc = (V + kCoarse - 1) / kCoarse;
    return ((sizeof(SharedM) + 15) & ~size_t(15)) + 2 * (size_t)nc * sizeof(float);
}

cudaError_t launch_mentor(const MentorParams& p, int grid, int resolve_grid, cudaStream_t stream) {
    const size_t smem = mentor_smem_bytes(p.V);
    auto kern = p.bf16 ? mentor_kernel<bf16_t> : mentor_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NT, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int rgrid = p.B < resolve_grid ? p.B : resolve_grid;
    (p.bf16 ? mentor_resolve_kernel<bf16_t> : mentor_resolve_kernel<float>)<<<rgrid, kDrawNT, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sv
