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
// draw. The bisection's result is the smallest dyadic alpha = j 2^-iters with
// KL(alpha) <= D. The sums above are needed only at the bisection's points, so
// a row is solved without sorting it (solve_hist: histograms of rho whose
// edges are the first ten levels, then exact sums over the few indices near
// alpha and beta); rows outside that scheme's limits take the sorting solve
// (solve: a stable LSD radix sort of ln(rho) in global scratch, the six
// running sums, and a multiway search evaluating up to 1023 grid points at a
// time). Rejections with alpha = 1 (beta = 1) and the bonus token use the
// verification path's own draw, so D = 0 reproduces spec_verify bit for bit.

#include "common.cuh"
#include "draw.cuh"

namespace sv {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int kIPT = 8;          // items per thread per sort tile
constexpr int kTile = NT * kIPT; // 8192
constexpr int kCoarse = 32;      // coarse index stride

// Large arrays of the sorting solve (dynamic shared memory, overlaid by the
// histogram solve's arrays: the two never run at the same time).
struct SharedM {
    uint32_t wcnt[NW][256];      // per-warp digit counts, then offsets
    uint32_t stk[kTile];         // one tile in digit order (keys, indices)
    uint32_t sti[kTile];
    uint32_t hist[4][256];       // all four digit histograms
    uint32_t base[256];          // next free global position per bucket
    uint32_t dtot[256];          // tile: per-digit count, start, global offset
    uint32_t dstart[256];
    uint32_t gofs[256];
};

// Small per-CTA state (static shared memory).
struct SmallM {
    double dred[NW];
    float wsum[5][NW];           // sorting solve: per-warp chunk totals
    float woff[5][NW];           //                and chunk offsets
    int ibuf[NW];
    int bi[8];
    double bd[8];
    long long wtot[3][NW];       // histogram solve: block scans
    long long wall[3];
    long long tA[3], tB[3];      // totals of the two histograms (q, p, q ln rho)
    long long base[3], above[3]; // sums below the alpha window, above the beta window
    long long ltot;              // sum of q ln rho over the row
    int hflag, ihi, inf, cnt, nA, n, a_b0, a_b1, b_lo, b_hi, ok;
    int iw[NW], scan_total;
    double ahi, abeta;
};

SV_DEV double block_sum_d(SmallM& s, double v) {
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
    float iSt, iSd;    // 1 / S, then corrected by the normalisation pass
    float lnr0, lnr0_lo;  // ln(iSt / iSd) as a sum of two floats
};

constexpr float kLn2 = 0.69314718055994531f;

// q, p and ln(q/p) of one index from its two logits: with a = z c2 - m c2
// (octaves below the maximum) q = 2^a_t iSt, p = 2^a_d iSd and
// ln(q/p) = ln 2 (a_t - a_d) + ln(iSt / iSd), so ln(q/p) is formed from the
// same exponents as q and p. The rounding of every step is pinned, so that
// the passes that recompute an index agree bit for bit.
template <typename E>
SV_DEV void qpl_of(const Row<E>& r, float zt, float zd, float& q, float& p, float& l) {
    const float at = __fmaf_rn(zt, r.c2, -r.mtc), ad = __fmaf_rn(zd, r.c2, -r.mdc);
    q = __fmul_rn(ex2(at), r.iSt);
    p = __fmul_rn(ex2(ad), r.iSd);
    l = __fadd_rn(__fmaf_rn(__fsub_rn(at, ad), kLn2, r.lnr0), r.lnr0_lo);
}

template <typename E>
SV_DEV void qpl(const Row<E>& r, int i, float& q, float& p, float& l) {
    qpl_of(r, VecTraits<E>::load1(r.rt + i), VecTraits<E>::load1(r.rd + i), q, p, l);
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
SV_DEV void solve(SharedM& s, SmallM& t, float* coarse, const MentorParams& p, const Row<E>& r, uint32_t* k0,
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
            float ql = (ok && q > 0.f) ? q * __ldcg(L + j) : 0.f;  // q = 0 contributes 0 (ln rho may be -inf)
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
            t.wsum[0][warp] = cq;
            t.wsum[1][warp] = cp;
            t.wsum[2][warp] = cl;
            t.wsum[3][warp] = sq;
            t.wsum[4][warp] = sp;
        }
    }
    __syncthreads();
    // chunk offsets in a fixed order: prefixes left to right, suffixes right to left
    if (tid < 5) {
        float acc = 0.f;
        if (tid < 3) {
            for (int w = 0; w < NW; ++w) {
                t.woff[tid][w] = acc;
                acc += t.wsum[tid][w];
            }
        } else {
            for (int w = NW - 1; w >= 0; --w) {
                t.woff[tid][w] = acc;
                acc += t.wsum[tid][w];
            }
        }
    }
    __syncthreads();
    {
        const float oq = t.woff[0][warp], op = t.woff[1][warp], ol = t.woff[2][warp];
        const float xq = t.woff[3][warp], xp = t.woff[4][warp];
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
        if ((tid & 31) == 0) t.ibuf[tid >> 5] = bal ? (tid + __ffs(bal) - 1) : 0x7FFFFFFF;
        __syncthreads();
        if (tid == 0) {
            int f = 0x7FFFFFFF;
            for (int w = 0; w < NW; ++w) f = min(f, t.ibuf[w]);
            t.bi[2] = f;
        }
        __syncthreads();
        const int f = t.bi[2];
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
            t.bd[0] = bt;
        }
        __syncthreads();
        *beta_out = (float)t.bd[0];
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Histogram solve: the same bisection without sorting the row.
//
// KL(alpha) needs, at alpha, the sums of q, p and q ln rho over {rho < alpha},
// and beta, where the decreasing function g(t) = sum_{rho >= t} (q/t - p)
// meets R = sum_{rho < alpha} (p - q/alpha); the indices with rho >= beta are
// the ones resampled from. alpha <= 1 <= beta always (at alpha = 1 both are
// 1), so one pass over the row builds two histograms:
//   * rho < 1: 1024 buckets of rho, width 2^-10, whose edges are the first
//     ten bisection levels, so the sums below a grid point are exact;
//   * rho >= 1: 4096 buckets of ln rho, width 1/128 (the last one open).
// The sums are 64-bit fixed point (q, p in units of 2^-50, q ln rho in
// 2^-46), so they are exact and independent of the order of the atomics.
//
// Round 0 evaluates the first bisection levels (up to 1023 grid points, one
// thread each, in fp32): beta is placed in its bucket exactly (g is known at
// every bucket edge), and the indices of that bucket are counted out of the
// resampled set. That choice is still a feasible redistribution of the
// rejected mass, so its KL is an upper bound of the true one, above it by at
// most Q_b d^2/2 (1 + Q_b/Q_U) for a bucket of q-mass Q_b and log-width d,
// plus the fp32 rounding of the three terms. Grid points whose bounds leave
// the comparison with D open are settled exactly below; KL falls as alpha
// grows, so they lie between the last surely infeasible point and the first
// surely feasible one.
//
// The exact evaluations (those points, the remaining bisection levels, and
// beta of the result) need only the indices whose rho falls in the alpha
// interval left by round 0 and the beta buckets that interval maps to: a second
// pass over the row (now in L2) collects them, they are sorted by ln rho in
// shared memory and summed exactly, and one warp searches the remaining levels
// 31 points at a time in double precision. Rows whose result lies below 2^-10,
// whose ambiguous range or windows are too large, or whose terms overflow the
// fixed point go to the sorting solve.
// ---------------------------------------------------------------------------
constexpr int kNA = 1024;             // alpha buckets of rho in [0, 1)
constexpr int kNB = 2048;             // beta buckets of ln rho in [0, 32) (last one open)
constexpr float kBScale = 64.f;       // beta buckets per unit of ln rho
constexpr int kCap = 2048;            // window indices
constexpr int kIdsSmem = 32768;       // rows up to this length keep their bucket ids in shared memory
constexpr int kMaxAmb = 64;           // grid points left open by round 0
constexpr float kQF = 0x1p44f, kLF = 0x1p40f;    // fixed-point scales of q, p and of q ln rho
constexpr float kQS = 0x1p-44f, kLS = 0x1p-40f;  // and their inverses
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaxAbsL = 65536.f;   // |ln rho| bound of the fixed point (q > 0)
constexpr uint32_t kDead = 0xFFFFu;   // bucket id of an index with q = p = 0

// A bucket's four 64-bit sums (q, p, and q ln rho split by sign) are kept as
// pairs of 32-bit words, added to with 32-bit shared atomics plus a carry
// (the value returned by the low word's atomic says whether it wrapped), then
// folded to three signed 64-bit sums in place by the scans. The scales keep
// almost every term below 2^32, so the high word is rarely touched.
constexpr int kWords = 8;
template <int N>
union HistSide {
    uint32_t raw[kWords][N];  // (lo, hi) of q, p, q ln rho >= 0, -(q ln rho > 0)
    long long s[3][N];        // after the scan: prefix (alpha) or suffix (beta) sums
};
struct HistArrays {
    HistSide<kNA> A;          // alpha buckets; then exclusive prefix sums
    HistSide<kNB> B;          // beta buckets; then inclusive suffix sums
    float gb[kNB];            // g at the lower edge of every beta bucket
    short bb[kNA + 8];        // round 0: first beta edge with g <= R per grid point
    uint16_t ids[kIdsSmem];   // pass 1: bucket id of every index (V <= kIdsSmem)
};
// Overlays HistArrays once round 0 is done. Pass 2 writes only `key`, which
// lies below `ids`; everything else is written after pass 2.
struct WinArrays {
    unsigned long long key[kCap];   // (ordered ln rho) << 32 | index, as collected
    unsigned long long skey[kCap];  // sorted
    long long c[3][kCap];           // alpha part: prefix sums; beta part: suffix sums
    float lw[kCap];                 // ln rho
    float gw[kCap];                 // beta part: g at each index's rho
    long long cu[3][kCap];          // the values in collection order
    float lwu[kCap];
};
union SharedH {
    HistArrays h;
    WinArrays w;
};

// x * scale (scale a power of two, 0 <= x scale < 2^56) rounded to the
// nearest integer, as 32-bit words: hi = floor(v / 2^32) and v - hi 2^32 are
// both exact in fp32, so two 32-bit conversions give the 64-bit integer.
struct Fix2 {
    uint32_t lo, hi;
};
SV_DEV Fix2 fix2(float x, float scale) {
    const float v = x * scale;
    const uint32_t hi = __float2uint_rd(v * 0x1p-32f);
    return {__float2uint_rn(fmaf(-(float)hi, 0x1p32f, v)), hi};
}

// Signed fixed point of x (|x| scale < 2^56).
SV_DEV long long to_fix(float x, float scale) {
    const Fix2 f = fix2(fabsf(x), scale);
    const long long v = (long long)(((unsigned long long)f.hi << 32) | f.lo);
    return x < 0.f ? -v : v;
}

// 64-bit integers to fp32 through two 32-bit conversions (about one rounding).
SV_DEV float ll2f(long long v) { return fmaf((float)(int)(v >> 32), 0x1p32f, __uint2float_rn((unsigned)v)); }
SV_DEV float ull2f(unsigned long long v) {
    return fmaf(__uint2float_rn((unsigned)(v >> 32)), 0x1p32f, __uint2float_rn((unsigned)v));
}
SV_DEV float fix_f(long long v, float scale) { return ll2f(v) * scale; }

// Adds f to the 64-bit sum held as (lo, hi) words.
SV_DEV void add64(uint32_t* lo, uint32_t* hi, Fix2 f) {
    uint32_t vh = f.hi;
    if (f.lo) {
        const uint32_t old = atomicAdd(lo, f.lo);
        vh += (old + f.lo < old) ? 1u : 0u;
    }
    if (vh) atomicAdd(hi, vh);
}

SV_DEV int alpha_bucket(float l) {  // l < 0
    const float rho = ex2(__fmul_rn(l, kLog2e));
    return min(kNA - 1, (int)__fmul_rn(rho, (float)kNA));
}

SV_DEV int beta_bucket(float l) {   // l >= 0, possibly +inf
    return l >= (float)kNB / kBScale ? kNB - 1 : (int)__fmul_rn(l, kBScale);
}

// Exclusive prefix over the 32 warps (in warp order) of three 64-bit warp
// totals, given on every lane; tot = the block totals.
SV_DEV void warp_offsets3(SmallM& t, long long (&v)[3], long long (&tot)[3]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 3; ++k) t.wtot[k][warp] = v[k];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const long long w0 = t.wtot[k][lane];
            long long w = w0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            t.wtot[k][lane] = w - w0;
            if (lane == 31) t.wall[k] = w;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        v[k] = t.wtot[k][warp];
        tot[k] = t.wall[k];
    }
    __syncthreads();
}

// Exclusive prefix in thread order of three 64-bit values; tot = totals.
SV_DEV void block_exscan3(SmallM& t, long long (&v)[3], long long (&tot)[3]) {
    const int lane = threadIdx.x & 31;
    long long inc[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const long long y = __shfl_up_sync(0xFFFFFFFFu, inc[k], o);
            if (lane >= o) inc[k] += y;
        }
    }
    long long wt[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) wt[k] = __shfl_sync(0xFFFFFFFFu, inc[k], 31);
    warp_offsets3(t, wt, tot);
#pragma unroll
    for (int k = 0; k < 3; ++k) v[k] = wt[k] + inc[k] - v[k];
}

// One index of pass 1: its bucket sums and its bucket id (alpha: 0..kNA-1,
// beta: kNA + bucket, kDead when q = p = 0).
template <typename E>
SV_DEV uint32_t hist_elem(HistArrays& h, const Row<E>& r, float zt, float zd, int& fl) {
    float q, p, l;
    qpl_of(r, zt, zd, q, p, l);
    if (!(q > 0.f) && !(p > 0.f)) return kDead;
    float ql = 0.f;
    if (q > 0.f) {
        if (l == INFINITY) {
            fl |= 1;
        } else if (!(fabsf(l) < kMaxAbsL)) {
            fl |= 2;
        } else {
            ql = __fmul_rn(q, l);
        }
    }
    uint32_t* H;
    int st;
    uint32_t id;
    if (l < 0.f) {
        const int j = alpha_bucket(l);
        if (!SV_IN(j, kNA)) return kDead;
        H = &h.A.raw[0][j];
        st = kNA;
        id = (uint32_t)j;
    } else {
        const int b = beta_bucket(l);
        if (!SV_IN(b, kNB)) return kDead;
        H = &h.B.raw[0][b];
        st = kNB;
        id = (uint32_t)(kNA + b);
    }
    if (q > 0.f) add64(H, H + st, fix2(q, kQF));
    if (p > 0.f) add64(H + 2 * st, H + 3 * st, fix2(p, kQF));
    if (ql > 0.f) add64(H + 4 * st, H + 5 * st, fix2(ql, kLF));
    if (ql < 0.f) add64(H + 6 * st, H + 7 * st, fix2(-ql, kLF));
    return id;
}

// Pass 1: both histograms of the row pair, and every index's bucket id in
// `ids` (16 bits per index, written with 8- or 16-byte stores). hflag bit 0:
// some index has q > 0 and p = 0 (KL(q || p) is infinite); bit 1: some index
// with q > 0 has |ln rho| too large for the fixed point.
template <typename E>
SV_DEV void hist_pass(HistArrays& h, SmallM& t, const Row<E>& r, int V, uint16_t* ids) {
    constexpr int kN = VecTraits<E>::kN;
    const int tid = threadIdx.x;
    for (int e = tid; e < kWords * kNA; e += NT) (&h.A.raw[0][0])[e] = 0u;
    for (int e = tid; e < kWords * kNB; e += NT) (&h.B.raw[0][0])[e] = 0u;
    const bool vec = ((reinterpret_cast<uintptr_t>(r.rt) | reinterpret_cast<uintptr_t>(r.rd)) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(ids) & (2 * kN - 1)) == 0;
    if (vec && tid < 4) {  // the row pair into L2 (bulk prefetch, 64 KB pieces)
        const size_t bytes = (size_t)(V / kN) * 16;
        const char* base = reinterpret_cast<const char*>(tid < 2 ? (const void*)r.rt : (const void*)r.rd);
        for (size_t o = (size_t)(tid & 1) * 65536; o < bytes; o += 131072) {
            const uint32_t sz = (uint32_t)(bytes - o < 65536 ? bytes - o : 65536);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(sz) : "memory");
        }
    }
    if (tid == 0) t.hflag = 0;
    __syncthreads();
    int fl = 0;
    int tail = 0;
    if (vec) {
        const int nv = V / kN;
        const uint4* vt = reinterpret_cast<const uint4*>(r.rt);
        const uint4* vd = reinterpret_cast<const uint4*>(r.rd);
        const auto proc = [&](int vv, const uint4& a, const uint4& b) {
            float x[kN], y[kN];
            VecTraits<E>::unpack(a, x);
            VecTraits<E>::unpack(b, y);
            uint32_t pk[kN / 2];
#pragma unroll
            for (int u = 0; u < kN; u += 2) {
                const uint32_t i0 = hist_elem(h, r, x[u], y[u], fl);
                const uint32_t i1 = hist_elem(h, r, x[u + 1], y[u + 1], fl);
                pk[u / 2] = i0 | (i1 << 16);
            }
            if constexpr (kN == 4) {
                *reinterpret_cast<uint2*>(ids + (size_t)vv * kN) = make_uint2(pk[0], pk[1]);
            } else {
                *reinterpret_cast<uint4*>(ids + (size_t)vv * kN) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        };
        for (int v = tid; v < nv; v += 2 * NT) {
            const bool two = v + NT < nv;
            const uint4 a0 = __ldg(vt + v), b0 = __ldg(vd + v);
            const uint4 a1 = two ? __ldg(vt + v + NT) : a0, b1 = two ? __ldg(vd + v + NT) : b0;
            proc(v, a0, b0);
            if (two) proc(v + NT, a1, b1);
        }
        tail = nv * kN;
    }
    for (int i = tail + tid; i < V; i += NT)
        ids[i] = (uint16_t)hist_elem(h, r, VecTraits<E>::load1(r.rt + i), VecTraits<E>::load1(r.rd + i), fl);
    if (fl) atomicOr(&t.hflag, fl);
    __syncthreads();
}

template <int N>
SV_DEV void bucket3(const HistSide<N>& H, int b, long long (&v)[3]) {
    const auto w64 = [&](int k) {
        return (long long)(((unsigned long long)H.raw[2 * k + 1][b] << 32) | H.raw[2 * k][b]);
    };
    v[0] = w64(0);
    v[1] = w64(1);
    v[2] = w64(2) - w64(3);
}

// Alpha buckets to exclusive prefix sums, beta buckets to inclusive suffix
// sums (both in place: every raw word is read before the first barrier of
// the block scans, every sum is written after it), totals, and g at every
// beta edge.
SV_DEV void scan_hist(HistArrays& h, SmallM& t) {
    const int tid = threadIdx.x;
    long long tot[3];
    {   // alpha: one bucket per thread
        long long v[3];
        bucket3(h.A, tid, v);
        block_exscan3(t, v, tot);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            h.A.s[k][tid] = v[k];
            if (tid == 0) t.tA[k] = tot[k];
        }
    }
    {   // beta: thread tid owns the two buckets [c0, c0 + 2), c0 = 2 (NT - 1 - tid),
        // so thread order is descending bucket order; 8- and 16-byte accesses
        static_assert(kNB == 2 * NT, "two beta buckets per thread");
        const int c0 = (NT - 1 - tid) * 2;
        long long sf[3][2];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint2 lo = *reinterpret_cast<const uint2*>(&h.B.raw[2 * k][c0]);
            const uint2 hi = *reinterpret_cast<const uint2*>(&h.B.raw[2 * k + 1][c0]);
            sf[k][0] = (long long)(((unsigned long long)hi.x << 32) | lo.x);
            sf[k][1] = (long long)(((unsigned long long)hi.y << 32) | lo.y);
        }
        {
            const uint2 lo = *reinterpret_cast<const uint2*>(&h.B.raw[6][c0]);
            const uint2 hi = *reinterpret_cast<const uint2*>(&h.B.raw[7][c0]);
            sf[2][0] -= (long long)(((unsigned long long)hi.x << 32) | lo.x);
            sf[2][1] -= (long long)(((unsigned long long)hi.y << 32) | lo.y);
        }
        long long v[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            sf[k][0] += sf[k][1];
            v[k] = sf[k][0];
        }
        block_exscan3(t, v, tot);  // v: the sums of all higher chunks
        float g[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int k = 0; k < 3; ++k) sf[k][u] += v[k];
            g[u] = fix_f(sf[0][u], kQS) * ex2(-(float)(c0 + u) * (kLog2e / kBScale)) - fix_f(sf[1][u], kQS);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            *reinterpret_cast<longlong2*>(&h.B.s[k][c0]) = make_longlong2(sf[k][0], sf[k][1]);
            if (tid == 0) t.tB[k] = tot[k];
        }
        *reinterpret_cast<float2*>(&h.gb[c0]) = make_float2(g[0], g[1]);
    }
    if (tid == 0) t.ltot = t.tA[2] + t.tB[2];
    __syncthreads();
}

// |n| as a float (about one rounding).
SV_DEV float i128_abs_f(__int128 n) {
    const unsigned __int128 u = n < 0 ? (unsigned __int128)(-n) : (unsigned __int128)n;
    return fmaf(ull2f((unsigned long long)(u >> 64)), 0x1p64f, ull2f((unsigned long long)u));
}

// The window search at alpha = J 2^-K: the sums below alpha, R exactly (as
// the integer (PL - QL/alpha) J = PL J - QL 2^K in fixed-point units), and
// the first window index of the resampled set.
struct WinEval {
    long long QL, PL, LL, QU, PU, LU;
    __int128 RJ;      // (PL - QL/alpha) J
    bool ok;          // the resampled set is not empty and R + PU > 0
};

SV_DEV WinEval win_eval(const WinArrays& w, const SmallM& t, uint64_t J, int K, float la) {
    WinEval e;
    int lo = 0, hi = t.nA;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (w.lw[mid] < la) lo = mid + 1; else hi = mid;
    }
    e.QL = lo ? w.c[0][lo - 1] : t.base[0];
    e.PL = lo ? w.c[1][lo - 1] : t.base[1];
    e.LL = lo ? w.c[2][lo - 1] : t.base[2];
    e.RJ = (__int128)e.PL * J - ((__int128)e.QL << K);
    const float R = (e.RJ < 0 ? -1.f : 1.f) * i128_abs_f(e.RJ) / ull2f(J) * kQS;
    lo = t.nA;
    hi = t.n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (w.gw[mid] <= R) hi = mid; else lo = mid + 1;
    }
    e.QU = lo < t.n ? w.c[0][lo] : t.above[0];
    e.PU = lo < t.n ? w.c[1][lo] : t.above[1];
    e.LU = lo < t.n ? w.c[2][lo] : t.above[2];
    e.ok = e.QU > 0 && e.RJ + (__int128)e.PU * J > 0;
    return e;
}

// ln(J 2^-K) in fp32: J = m 2^e with m in [1/2, 1), so the log is
// ln m + (e - K) ln 2 without cancellation, and the rounding of J to fp32 is
// corrected to first order.
SV_DEV float ln_grid(uint64_t J, int K) {
    const float jf = ull2f(J);
    const float res = ll2f((long long)(J - (uint64_t)jf));  // J - jf
    int e;
    const float m = frexpf(jf, &e);
    return logf(m) + (float)(e - K) * 0.69314718055994531f + res / jf;
}

// KL(alpha) from the windows in fp32 (the sums are exact integers, R is
// exact before its one rounding); +inf when the resampled set is empty.
SV_DEV float kl_win(const WinArrays& w, const SmallM& t, uint64_t J, int K) {
    const float la = ln_grid(J, K);
    const WinEval e = win_eval(w, t, J, K, la);
    if (!e.ok) return INFINITY;
    const __int128 den = e.RJ + (__int128)e.PU * J;  // (R + PU) J, fixed-point units
    const float beta = ll2f(e.QU) * ull2f(J) / i128_abs_f(den);
    return la * fix_f(e.QL, kQS) + fix_f(t.ltot - e.LL - e.LU, kLS) + logf(beta) * fix_f(e.QU, kQS);
}

// n as a double (about one rounding).
SV_DEV double i128_d(__int128 n) {
    const bool neg = n < 0;
    const unsigned __int128 u = neg ? (unsigned __int128)(-n) : (unsigned __int128)n;
    const double d = (double)(unsigned long long)(u >> 64) * 0x1p64 + (double)(unsigned long long)u;
    return neg ? -d : d;
}

// beta at alpha = J 2^-K, in double (one division).
SV_DEV double beta_win(const WinArrays& w, const SmallM& t, uint64_t J, int K) {
    const WinEval e = win_eval(w, t, J, K, ln_grid(J, K));
    if (!e.ok) return 1.0;
    return i128_d((__int128)e.QU * J) / i128_d(e.RJ + (__int128)e.PU * J);
}

// Returns false when the row has to go to the sorting solve.
template <typename E>
SV_DEV bool solve_hist(SharedH& sh, SmallM& t, const MentorParams& p, const Row<E>& r, const uint16_t* ids,
                       double* alpha_out, float* beta_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = p.V;
    const float D = p.kl_bound;
    const int bits0 = min(10, p.iters), npts = 1 << bits0, stp = kNA >> bits0;
    const bool rounds = p.iters > bits0;
    HistArrays& h = sh.h;
    // round 0
    if (tid == 0) {
        t.ihi = npts;
        t.inf = 0;
        h.bb[0] = (short)kNB;  // alpha -> 0: beta above every edge
        h.bb[npts] = 0;        // alpha = 1: beta = 1, bucket 0
    }
    __syncthreads();
    const int i = tid + 1;
    bool maybe = true;
    if (i < npts) {
        const int j = i * stp;
        const float a = (float)j * (1.f / kNA);
        const long long QLi = h.A.s[0][j], PLi = h.A.s[1][j], LLi = h.A.s[2][j];
        const long long RJ = PLi * j - QLi * kNA;  // (PL - QL/a) j, exact
        const float R = ll2f(RJ) / (float)j * kQS;
        int lo = 0, hi = kNB;  // first edge with g <= R (kNB: none)
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (h.gb[mid] <= R) hi = mid; else lo = mid + 1;
        }
        const int b = lo;
        h.bb[i] = (short)b;
        bool sure = false;
        if (b < kNB && h.B.s[0][b] > 0 && RJ + h.B.s[1][b] * j > 0) {
            const float QU = fix_f(h.B.s[0][b], kQS);
            // QU / (R + PU) with both sides in fixed-point units
            const float beta = ll2f(h.B.s[0][b]) * (float)j / ll2f(RJ + h.B.s[1][b] * j);
            const float QL = fix_f(QLi, kQS);
            const float LM = fix_f(t.ltot - LLi - h.B.s[2][b], kLS);
            const float t1 = logf(a) * QL, t3 = logf(beta) * QU;
            const float kl = t1 + LM + t3;
            const float QB = b > 0 ? fix_f(h.B.s[0][b - 1] - h.B.s[0][b], kQS) : 0.f;
            const float efp = 4e-7f * (fabsf(t1) + fabsf(LM) + fabsf(t3)) + 1e-9f;
            const float err = QB * (0.5f / (kBScale * kBScale)) * (1.f + QB / QU) * 1.01f + efp;
            sure = kl + efp <= D;
            maybe = !(kl - err > D);
        }
        if (sure) atomicMin(&t.ihi, i);
    }
    __syncthreads();
    if (i < t.ihi && !maybe) atomicMax(&t.inf, i);
    __syncthreads();
    if (tid == 0) {
        const int ihi = t.ihi, ilo = t.inf + 1;
        const bool ok = !(t.hflag & 2) && !(rounds && ilo == 1) && ihi - ilo <= kMaxAmb;
        t.inf = ilo;
        t.cnt = 0;
        t.nA = 0;
        t.ok = ok;
        if (ok) {
            // every grid point in [ilo - 1, ihi] was evaluated above (bb
            // holds its beta edge); clamps keep the indexes in range
            const int a_b0 = (rounds ? ilo - 1 : ilo) * stp, a_b1 = ihi * stp;
            const int b_lo = ihi < npts ? max(0, (int)h.bb[ihi] - 2) : 0;
            const int b_hi = max(0, min(kNB - 1, (int)h.bb[rounds ? ilo - 1 : ilo]));
            t.a_b0 = a_b0;
            t.a_b1 = a_b1;
            t.b_lo = b_lo;
            t.b_hi = b_hi;
            for (int k = 0; k < 3; ++k) {
                t.base[k] = a_b0 < kNA ? h.A.s[k][a_b0] : t.tA[k];
                t.above[k] = b_hi + 1 < kNB ? h.B.s[k][b_hi + 1] : 0;
            }
        }
    }
    __syncthreads();
    if (!t.ok) return false;
    const int ilo = t.inf, ihi = t.ihi;
    if (!rounds && ilo == ihi && ihi == npts) {  // alpha = 1 (every grid point below is infeasible)
        *alpha_out = 1.0;
        *beta_out = 1.f;
        return true;
    }
    // pass 2: the window indices, from the bucket ids of pass 1. Each thread
    // counts its candidates, a block scan gives it its output offset, and a
    // second walk writes them (ordered by thread, no atomics).
    WinArrays& w = sh.w;
    {
        const uint32_t A0 = (uint32_t)t.a_b0, A1 = (uint32_t)t.a_b1;
        const uint32_t B0 = (uint32_t)(kNA + t.b_lo), B1 = (uint32_t)(kNA + t.b_hi);
        const auto sel = [&](uint32_t id) { return id < (uint32_t)kNA ? (id >= A0 && id < A1) : (id >= B0 && id <= B1); };
        // one walk over the ids: each warp appends its candidates to a private
        // buffer (ballot ranks, no atomics; warp order, then index order), a
        // scan of the 32 warp counts places the buffers. The buffers live in
        // `skey`, which is free until the sort and lies below the ids.
        constexpr int kWarpBuf = kCap * 2 / NW;  // 32-bit entries per warp
        uint32_t* wb = reinterpret_cast<uint32_t*>(w.skey) + warp * kWarpBuf;
        const unsigned lt = (1u << lane) - 1u;
        const auto collect = [&](const uint16_t* idp) {
            const bool vec = (reinterpret_cast<uintptr_t>(idp) & 15u) == 0;
            const int n8 = vec ? V / 8 : 0;
            const uint4* iv = reinterpret_cast<const uint4*>(idp);
            int wc = 0;
            for (int v0 = warp * 32; v0 < n8; v0 += NT) {  // warp-uniform trip count
                const int v = v0 + lane;
                const bool ok = v < n8;
                const uint4 x = ok ? iv[v] : make_uint4(kDead | (kDead << 16), kDead | (kDead << 16),
                                                        kDead | (kDead << 16), kDead | (kDead << 16));
                const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const bool pr = sel(c & 1 ? wd[c >> 1] >> 16 : wd[c >> 1] & 0xFFFFu);
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, pr);
                    if (pr) {
                        const int pos = wc + __popc(bal & lt);
                        if (pos < kWarpBuf) wb[pos] = (uint32_t)(v * 8 + c);
                    }
                    wc += __popc(bal);
                }
            }
            for (int i0 = n8 * 8 + warp * 32; i0 < V; i0 += NT) {
                const int idx = i0 + lane;
                const bool pr = idx < V && sel(idp[idx]);
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, pr);
                if (pr) {
                    const int pos = wc + __popc(bal & lt);
                    if (pos < kWarpBuf) wb[pos] = (uint32_t)idx;
                }
                wc += __popc(bal);
            }
            return wc;
        };
        const int wc = V <= kIdsSmem ? collect(sh.h.ids) : collect(ids);
        if (lane == 0) t.iw[warp] = wc;
        __syncthreads();
        if (warp == 0) {
            const int c0 = t.iw[lane];
            int c = c0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, c, o);
                if (lane >= o) c += y;
            }
            t.iw[lane] = c - c0;
            const bool over = __any_sync(0xFFFFFFFFu, c0 > kWarpBuf);
            if (lane == 31) t.scan_total = over ? kCap + 1 : c;
        }
        __syncthreads();
        const int off = t.iw[warp];
        for (int i = lane; i < wc && i < kWarpBuf; i += 32)
            if (off + i < kCap) w.key[off + i] = wb[i];
    }
    __syncthreads();
    const int n = t.scan_total;
    if (n > kCap) return false;
    // keys and values of the window indices (recomputed exactly as in pass 1)
    for (int s = tid; s < n; s += NT) {
        const int idx = (int)(uint32_t)w.key[s];
        float q, pp, l;
        qpl(r, idx, q, pp, l);
        const float ql = (q > 0.f && l != INFINITY) ? __fmul_rn(q, l) : 0.f;
        w.key[s] = ((unsigned long long)f32_key(l) << 32) | (unsigned)idx;
        w.cu[0][s] = q > 0.f ? to_fix(q, kQF) : 0;
        w.cu[1][s] = pp > 0.f ? to_fix(pp, kQF) : 0;
        w.cu[2][s] = ql != 0.f ? to_fix(ql, kLF) : 0;
        w.lwu[s] = l;
    }
    __syncthreads();
    if (n <= NT) {
        // keys (ordered ln rho) << 32 | collection slot (the collection order
        // is deterministic, so ties in ln rho are too). Each warp sorts a run
        // of 32 keys in registers; a key's rank is its place in its run plus
        // the count of smaller keys in every other run (binary searches), and
        // its values are placed from its slot.
        int n2 = 32;
        while (n2 < n) n2 <<= 1;
        const int runs = n2 / 32;
        const bool wact = warp < runs;
        unsigned long long x = ~0ull;
        if (tid < n) x = (w.key[tid] & 0xFFFFFFFF00000000ull) | (unsigned)tid;
        if (wact) {
#pragma unroll
            for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
                for (int j = k >> 1; j > 0; j >>= 1) {
                    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
                    const bool keep_min = ((lane & j) == 0) == ((lane & k) == 0);
                    if ((y < x) == keep_min) x = y;
                }
            }
            w.skey[tid] = x;  // run `warp`, ascending
        }
        __syncthreads();
        if (wact && x != ~0ull) {
            int rank = lane;
            for (int rr = 0; rr < runs; ++rr) {
                if (rr == warp) continue;
                const unsigned long long* run = w.skey + rr * 32;
                int pos = 0;
#pragma unroll
                for (int st = 16; st; st >>= 1)
                    if (run[pos + st - 1] < x) pos += st;
                pos += run[pos] < x ? 1 : 0;
                rank += pos;
            }
            const int slot = (int)(uint32_t)x;
            if (SV_IN(rank, kCap) && SV_IN(slot, kCap)) {
#pragma unroll
                for (int k = 0; k < 3; ++k) w.c[k][rank] = w.cu[k][slot];
                w.lw[rank] = w.lwu[slot];
            }
            if ((uint32_t)(x >> 32) < 0x80000000u) atomicAdd(&t.nA, 1);
        }
    } else {
        int n2 = 2;
        while (n2 < n) n2 <<= 1;
        for (int s = n + tid; s < n2; s += NT) w.key[s] = ~0ull;
        __syncthreads();
        for (int k = 2; k <= n2; k <<= 1) {
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
                for (int x = tid; x < n2; x += NT) {
                    const int y = x ^ jj;
                    if (y > x) {
                        const unsigned long long ka = w.key[x], kb = w.key[y];
                        if ((ka > kb) == ((x & k) == 0)) {
                            w.key[x] = kb;
                            w.key[y] = ka;
                        }
                    }
                }
                __syncthreads();
            }
        }
        for (int s = tid; s < n; s += NT) {
            w.skey[s] = w.key[s];
            if ((uint32_t)(w.key[s] >> 32) < 0x80000000u) atomicAdd(&t.nA, 1);
        }
    }
    if (tid == 0) t.n = n;
    __syncthreads();
    // the window's values in sorted order (already placed by the run sort;
    // after the shared-memory sort, recomputed exactly as in pass 1)
    for (int s = tid; n > NT && s < n; s += NT) {
        const int idx = (int)(uint32_t)w.skey[s];
        float q, pp, l;
        qpl(r, idx, q, pp, l);
        const float ql = (q > 0.f && l != INFINITY) ? __fmul_rn(q, l) : 0.f;
        w.c[0][s] = q > 0.f ? to_fix(q, kQF) : 0;
        w.c[1][s] = pp > 0.f ? to_fix(pp, kQF) : 0;
        w.c[2][s] = ql != 0.f ? to_fix(ql, kLF) : 0;
        w.lw[s] = l;
    }
    __syncthreads();
    // alpha part [0, nA): inclusive prefix sums from base; beta part [nA, n):
    // inclusive suffix sums from above. Warps 0-2 and 3-5, one sum each.
    if (warp < 6) {
        const int k = warp % 3;
        const bool suf = warp >= 3;
        const int s0 = suf ? t.nA : 0, s1 = suf ? n : t.nA;
        const int per = (s1 - s0 + 31) / 32;
        const int c0 = suf ? max(s0, s1 - (lane + 1) * per) : min(s1, s0 + lane * per);
        const int c1 = suf ? max(s0, s1 - lane * per) : min(s1, c0 + per);
        long long sum = 0;
        for (int x = c0; x < c1; ++x) sum += w.c[k][x];
        long long inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
        }
        long long run = (suf ? t.above[k] : t.base[k]) + inc - sum;
        if (!suf) {
            for (int x = c0; x < c1; ++x) {
                run += w.c[k][x];
                w.c[k][x] = run;
            }
        } else {
            for (int x = c1 - 1; x >= c0; --x) {
                run += w.c[k][x];
                w.c[k][x] = run;
            }
        }
    }
    __syncthreads();
    for (int s = t.nA + tid; s < n; s += NT)
        w.gw[s] = fix_f(w.c[0][s], kQS) * ex2(-w.lw[s] * kLog2e) - fix_f(w.c[1][s], kQS);
    __syncthreads();
    // exact search on the dyadic grid alpha = J 2^-K: the open points of
    // round 0 (warp 0), then the remaining levels, up to 1023 points at a time
    if (warp == 0) {
        int it = ihi;
        for (int b0 = ilo; b0 < ihi; b0 += 32) {
            const int ii = b0 + lane;
            const bool f = ii < ihi && kl_win(w, t, (uint64_t)(ii * stp), 10) <= D;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, f);
            if (bal) {
                it = b0 + __ffs(bal) - 1;
                break;
            }
        }
        if (lane == 0) t.inf = it;
    }
    __syncthreads();
    // hi = J 2^-K; each level adds bits to K. Levels beyond 2^-60 move alpha
    // by less than its double-precision resolution near 1/2 and are not taken.
    uint64_t J = (uint64_t)(t.inf * stp);
    int K = 10;
    for (int left = min(p.iters, 60) - bits0; left > 0;) {
        const int bits = min(10, left), nn = 1 << bits;
        J <<= bits;
        K += bits;
        const uint64_t lo = J - (uint64_t)nn;  // hi - one step of the previous level
        if (tid == 0) t.cnt = nn;
        __syncthreads();
        if (i < nn && kl_win(w, t, lo + (uint64_t)i, K) <= D) atomicMin(&t.cnt, i);
        __syncthreads();
        if (t.cnt < nn) J = lo + (uint64_t)t.cnt;
        left -= bits;
        __syncthreads();
    }
    if (tid == 0) {
        const double a = ldexp((double)J, -K);
        t.ahi = a;
        t.abeta = a < 1.0 ? beta_win(w, t, J, K) : 1.0;
    }
    __syncthreads();
    if (tid == 0) {  // the caller reads the result on thread 0 only
        *alpha_out = t.ahi;
        *beta_out = (float)t.abeta;
    }
    return true;
}

// The sorting solve's input: sort keys of ln rho, indices, and q, p, ln rho
// per index in the scratch arrays; returns KL(q || p).
template <typename E>
SV_DEV double sort_pass(SmallM& t, const Row<E>& r, int V, uint32_t* k0, uint32_t* i0, float* A) {
    float acc_kl = 0.f;
    for (int i = threadIdx.x; i < V; i += NT) {
        float qq, pp, l;
        qpl(r, i, qq, pp, l);
        if (!(qq > 0.f) && !(pp > 0.f)) l = -INFINITY;  // q = p = 0: rho = 0 (ln rho would be NaN)
        if (qq > 0.f) acc_kl += qq * l;
        k0[i] = f32_key(l);
        i0[i] = (uint32_t)i;
        A[V + i] = qq;
        A[2 * (size_t)V + i] = pp;
        A[3 * (size_t)V + i] = l;
    }
    return block_sum_d(t, (double)acc_kl);
}

// Normalisation pass over the row pair, before a solve: the exact
// fixed-point totals of q and p as every later pass computes them (q, p in
// units of 2^-44, the histogram's units), then iSt and iSd are rescaled so
// that both totals are one, and ln(iSt / iSd) is formed in double from the
// rescaled floats. The rows' normalisers S come from fp32 sums and the
// rounding of m c2, which leave a common relative error of order 1e-7 to
// 1e-6 in every q and p; the bisection's alpha moves with such an error
// about ten times as much (the KL bound is met at a slope of order D), so
// the solve works with sums that are exact for the values it uses.
template <typename E>
SV_DEV void normalise(SmallM& t, Row<E>& r, int V) {
    constexpr int kN = VecTraits<E>::kN;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long sq = 0ull, sp = 0ull;
    const auto add = [&](float zt, float zd) {
        const float q = __fmul_rn(ex2(__fmaf_rn(zt, r.c2, -r.mtc)), r.iSt);
        const float p = __fmul_rn(ex2(__fmaf_rn(zd, r.c2, -r.mdc)), r.iSd);
        if (q > 0.f) {
            const Fix2 f = fix2(q, kQF);
            sq += ((unsigned long long)f.hi << 32) | f.lo;
        }
        if (p > 0.f) {
            const Fix2 f = fix2(p, kQF);
            sp += ((unsigned long long)f.hi << 32) | f.lo;
        }
    };
    int tail = 0;
    if (((reinterpret_cast<uintptr_t>(r.rt) | reinterpret_cast<uintptr_t>(r.rd)) & 15u) == 0) {
        const int nv = V / kN;
        const uint4* vt = reinterpret_cast<const uint4*>(r.rt);
        const uint4* vd = reinterpret_cast<const uint4*>(r.rd);
        for (int v = tid; v < nv; v += 2 * NT) {
            const bool two = v + NT < nv;
            const uint4 a0 = __ldg(vt + v), b0 = __ldg(vd + v);
            const uint4 a1 = two ? __ldg(vt + v + NT) : a0, b1 = two ? __ldg(vd + v + NT) : b0;
            float x[kN], y[kN];
            VecTraits<E>::unpack(a0, x);
            VecTraits<E>::unpack(b0, y);
#pragma unroll
            for (int u = 0; u < kN; ++u) add(x[u], y[u]);
            if (two) {
                VecTraits<E>::unpack(a1, x);
                VecTraits<E>::unpack(b1, y);
#pragma unroll
                for (int u = 0; u < kN; ++u) add(x[u], y[u]);
            }
        }
        tail = nv * kN;
    }
    for (int i = tail + tid; i < V; i += NT) add(VecTraits<E>::load1(r.rt + i), VecTraits<E>::load1(r.rd + i));
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
        sp += __shfl_xor_sync(0xFFFFFFFFu, sp, o);
    }
    if (lane == 0) {
        t.wtot[0][warp] = (long long)sq;
        t.wtot[1][warp] = (long long)sp;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long Q = 0ull, P = 0ull;
        for (int w = 0; w < NW; ++w) {
            Q += (unsigned long long)t.wtot[0][w];
            P += (unsigned long long)t.wtot[1][w];
        }
        // both totals are positive (the row maximum has q = 1/S > 0)
        const float ist = Q ? (float)((double)r.iSt * 0x1p44 / (double)Q) : r.iSt;
        const float isd = P ? (float)((double)r.iSd * 0x1p44 / (double)P) : r.iSd;
        const double l0 = log((double)ist) - log((double)isd);
        const float hi = (float)l0;
        t.bd[0] = (double)ist;
        t.bd[1] = (double)isd;
        t.bd[2] = (double)hi;
        t.bd[3] = (double)(float)(l0 - (double)hi);
    }
    __syncthreads();
    r.iSt = (float)t.bd[0];
    r.iSd = (float)t.bd[1];
    r.lnr0 = (float)t.bd[2];
    r.lnr0_lo = (float)t.bd[3];
    __syncthreads();
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
    __shared__ SmallM sm;
    SharedM& s = *reinterpret_cast<SharedM*>(smem_raw);
    SharedH& sh = *reinterpret_cast<SharedH*>(smem_raw);
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
    // pass-1 bucket ids: shared memory for rows up to kIdsSmem, else global
    // scratch (which the sorting solve reuses afterwards)
    uint16_t* ids = V <= kIdsSmem ? sh.h.ids : reinterpret_cast<uint16_t*>(k0);
    const E* tgt = reinterpret_cast<const E*>(p.target);
    const E* dft = reinterpret_cast<const E*>(p.draft);
    const long long jobs = (long long)p.B * G;

    for (;;) {
        if (tid == 0) sm.bi[4] = (int)atomicAdd(p.work, 1u);
        __syncthreads();
        const long long job = sm.bi[4];
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
        if (tid == 0) sm.bi[5] = G - (int)__ldcg(p.rejmark + b) < k;
        __syncthreads();
        const bool skip = sm.bi[5] != 0;
        __syncthreads();
        if (bad || skip) continue;

        // the verification path's probabilities and standard test
        const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
        float alpha = -1.f, beta = 0.f;
        int state = accept_test(u, q, pd) ? kPosAccepted : kPosRejected;
        float iS[2] = {1.f / t.S, 1.f / d.S};
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
            normalise<E>(sm, r, V);
            iS[0] = r.iSt;
            iS[1] = r.iSd;
            // KL(q || p) from the histogram pass (exact sum of the fp32 terms)
            if (V <= kIdsSmem) hist_pass<E>(sh.h, sm, r, V, sh.h.ids); else hist_pass<E>(sh.h, sm, r, V, ids);
            scan_hist(sh.h, sm);
            // (double precision is scarce on this part: thread 0 takes the
            // scalar decisions in double and shares them)
            const bool big = (sm.hflag & 2) != 0;
            if (tid == 0)
                sm.bi[6] = !big && !(sm.hflag & 1) && (double)sm.ltot * (double)kLS <= (double)p.kl_bound;
            __syncthreads();
            bool shortcut = sm.bi[6] != 0;
            if (big) shortcut = sort_pass<E>(sm, r, V, k0, i0, A) <= (double)p.kl_bound;
            if (shortcut) {
                state = kPosAccepted;
                alpha = 0.f;
            } else {
                double a = 1.0;
                beta = 1.f;
                if (p.kl_bound > 0.f && (big || !solve_hist<E>(sh, sm, p, r, ids, &a, &beta))) {
                    if (!big) sort_pass<E>(sm, r, V, k0, i0, A);
                    __threadfence_block();
                    __syncthreads();
                    solve<E>(s, sm, coarse, p, r, k0, i0, k1, i1, A, &a, &beta);
                }
                if (tid == 0) {
                    alpha = (float)a;
                    // alpha = 1 is the standard test, which failed
                    if (a < 1.0) {
                        const double rho = pd > 0.f ? (double)q / (double)pd : (q > 0.f ? HUGE_VAL : 0.0);
                        state = (double)u < fmin(1.0, rho / a) ? kPosAccepted : kPosRejectedScaled;
                    }
                }
            }
        }
        if (tid == 0 && SV_IN_SEQ(pos, (long long)p.B * G, p.status, b)) {
            if (p.alpha_out) p.alpha_out[pos] = alpha;
            if (p.beta_out) p.beta_out[pos] = beta;
            p.pos_beta[pos] = beta;
            p.pos_scale[2 * pos] = iS[0];
            p.pos_scale[2 * pos + 1] = iS[1];
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
                    // max(0, q/beta - p) with the q and p the solve normalised
                    const float beta = __ldcg(p.pos_beta + (size_t)b * G + n);
                    const float ist = __ldcg(p.pos_scale + 2 * ((size_t)b * G + n));
                    const float isd = __ldcg(p.pos_scale + 2 * ((size_t)b * G + n) + 1);
                    const ResidualW w{KeptExp{t.thr, c2, t.m * c2, ist * (1.f / beta)},
                                      KeptExp{d.thr, c2, d.m * c2, isd}};
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
            if (SV_IN_SEQ((size_t)b * G1 + j, (long long)p.B * G1, p.status, b)) p.tokens[(size_t)b * G1 + j] = v;
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
    const size_t sorting = ((sizeof(SharedM) + 15) & ~size_t(15)) + 2 * (size_t)nc * sizeof(float);
    return sorting > sizeof(SharedH) ? sorting : sizeof(SharedH);
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

SV_DEBUG_READER(mentor)

}  // namespace sv
