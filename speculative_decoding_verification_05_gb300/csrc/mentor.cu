// Mentor (lossy) verification, second stage.
//
// "推测解码的一种最优有损变体", section "解决优化问题": the KL-bounded optimum
// has r_i = min(1, q_i/(alpha p_i)) and s_i ~ max(0, q_i/beta - p_i), with KL
// falling as alpha grows, so alpha is found by bisection; the page lists the
// savings used here: only positions whose uniform fails the standard test
// u < min(1, q/p) are solved (the row kernel already decided the others), a
// row with KL(q || p) <= D is accepted directly, and the six running sums
// over the indices sorted by rho = q/p are computed once per row:
//   cq = sum_{i<=j} q, cp = sum_{i<=j} p, sq = sum_{i>=j} q, sp = sum_{i>=j} p,
//   cl = sum_{i<=j} q ln(q/p), g = (p_j/q_j) sq_j - sp_j.
// For alpha: k = #{rho < alpha}, R = cp_{k-1} - cq_{k-1}/alpha, m = first j
// with g_j <= R, beta = sq_m/(R + sp_m) and
//   KL(alpha) = ln(alpha) cq_{k-1} + (cl_{m-1} - cl_{k-1}) + ln(beta) sq_m.
//
// One CTA (1024 threads) per solved position, persistent over positions.
// The sort is a stable LSD radix sort (four 8-bit digit passes) of the fp32
// keys of ln(rho) in global scratch. The bisection's result (the smallest
// dyadic alpha = j 2^-iters with KL(alpha) <= D) is found by a multiway
// search: each round evaluates KL at up to 1023 interior grid points of the
// current interval in parallel, ten bisection steps at a time.

#include "common.cuh"

namespace sv {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int kIPT = 8;          // items per thread per sort tile
constexpr int kTile = NT * kIPT; // 8192
constexpr int kCoarse = 32;      // coarse index stride

struct SharedM {
    uint32_t wcnt[NW][256];      // per-warp digit counts, then offsets
    uint32_t base[256];
    double dred[NW];
    float fred[NW];
    float warp_tot[NW];
    float warp_pre[NW + 1];
    int ibuf[NW];
    int bi[8];
    float bf[8];
    double bd[8];
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

// Inclusive scan over the flattened order (thread chunks in thread order),
// sequential inside each thread and warp, so every running sum is an ordinary
// left-to-right sum of the previous partial sums. Returns the thread's
// exclusive prefix.
SV_DEV float block_excl(SharedM& s, float thr_sum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float wt;
    const float lp = warp_seq_exclusive(thr_sum, &wt);
    if (lane == 0) s.warp_tot[warp] = wt;
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int w = 0; w < NW; ++w) {
            s.warp_pre[w] = acc;
            acc += s.warp_tot[w];
        }
        s.warp_pre[NW] = acc;
    }
    __syncthreads();
    const float r = s.warp_pre[warp] + lp;
    __syncthreads();
    return r;
}

struct Row {
    const void* rt;    // target / draft rows (fp32 or bf16)
    const void* rd;
    int bf16;
    float mtc, mdc;    // m * c2
    float c2, inv_t;
    float iSt, iSd;    // 1 / S
    float lnr0;        // -(m_t - m_d)/T - ln S_t + ln S_d
};

SV_DEV float load_logit(const void* row, int bf16, int i) {
    if (bf16) {
        const unsigned short v = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
        return __uint_as_float(((uint32_t)v) << 16);
    }
    return __ldg(reinterpret_cast<const float*>(row) + i);
}

SV_DEV void qpl(const Row& r, int i, float& q, float& p, float& l) {
    const float zt = load_logit(r.rt, r.bf16, i), zd = load_logit(r.rd, r.bf16, i);
    q = ex2(fmaf(zt, r.c2, -r.mtc)) * r.iSt;
    p = ex2(fmaf(zd, r.c2, -r.mdc)) * r.iSd;
    l = (zt - zd) * r.inv_t + r.lnr0;
}

// Stable LSD radix sort of (key, idx) pairs, ascending, four 8-bit digits.
// k0/i0 hold the input; the sorted result ends in k0/i0 again.
SV_DEV void radix_sort(SharedM& s, uint32_t* k0, uint32_t* i0, uint32_t* k1, uint32_t* i1, int n) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 8 * pass;
        uint32_t* sk = pass & 1 ? k1 : k0;
        uint32_t* si = pass & 1 ? i1 : i0;
        uint32_t* dk = pass & 1 ? k0 : k1;
        uint32_t* di = pass & 1 ? i0 : i1;
        // digit histogram -> exclusive bucket starts
        for (int d = tid; d < 256; d += NT) s.base[d] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += NT) atomicAdd(&s.base[(__ldcg(sk + i) >> shift) & 255u], 1u);
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], seg = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = s.base[lane * 8 + j];
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
        // stable scatter, tile by tile; warp w owns items [w*256, w*256+256) of a tile
        for (int t0 = 0; t0 < n; t0 += kTile) {
            for (int e = tid; e < NW * 256; e += NT) (&s.wcnt[0][0])[e] = 0u;
            __syncthreads();
            uint32_t key[kIPT], idv[kIPT], rank[kIPT];
            int dig[kIPT];
#pragma unroll
            for (int r = 0; r < kIPT; ++r) {
                const int i = t0 + warp * (32 * kIPT) + r * 32 + lane;
                const bool ok = i < n;
                key[r] = ok ? __ldcg(sk + i) : 0u;
                idv[r] = ok ? __ldcg(si + i) : 0u;
                dig[r] = ok ? (int)((key[r] >> shift) & 255u) : -1;
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
            // offsets: digit-major over warps, starting at the bucket's running base
            {
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
                const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 3, 4);
                const uint32_t b0 = s.base[d];
                uint32_t run = b0 + incl - sum;
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    s.wcnt[q * 8 + j][d] = run;
                    run += c[j];
                }
                if (q == 3) s.base[d] = b0 + total;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kIPT; ++r) {
                if (dig[r] >= 0) {
                    const uint32_t pos = s.wcnt[warp][dig[r]] + rank[r];
                    dk[pos] = key[r];
                    di[pos] = idv[r];
                }
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
    const int k = count_less(a, log(alpha));
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
    return log(alpha) * qlow + lmid + log(beta) * sqm;
}

// Inverse-CDF draw in index order over weights w(i), one CTA; the smallest i
// with C_i > u W, or the last positive weight if rounding leaves none.
template <typename WF>
SV_DEV int block_draw(SharedM& s, int n, float u, WF wfun, float* W_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + NT - 1) / NT;
    const int i0 = tid * per, i1 = min(n, i0 + per);
    float tw = 0.f;
    for (int i = i0; i < i1; ++i) tw += wfun(i);
    float wt;
    const float lp = warp_seq_exclusive(tw, &wt);
    if (lane == 0) s.warp_tot[warp] = wt;
    __syncthreads();
    if (tid == 0) {
        float acc = 0.f;
        for (int w = 0; w < NW; ++w) {
            s.warp_pre[w] = acc;
            acc += s.warp_tot[w];
        }
        s.warp_pre[NW] = acc;
        const float t = u * acc;
        int ow = -1;
        for (int w = 0; w < NW; ++w)
            if (s.warp_pre[w] <= t && s.warp_tot[w] > 0.f) ow = w;
        s.bi[0] = ow;
        s.bi[1] = -1;
        s.bf[0] = acc;
        s.bf[1] = ow >= 0 ? t - s.warp_pre[ow] : 0.f;
    }
    __syncthreads();
    const int ow = s.bi[0];
    if (warp == ow) {
        const float tw_ = s.bf[1];
        const unsigned m = __ballot_sync(0xFFFFFFFFu, lp <= tw_ && tw > 0.f);
        const int ol = m ? 31 - __clz(m) : -1;
        if (lane == ol) {
            const float tt = tw_ - lp;
            float acc = 0.f;
            int found = -1, lastpos = -1;
            for (int i = i0; i < i1; ++i) {
                const float w = wfun(i);
                if (w > 0.f) lastpos = i;
                acc += w;
                if (w > 0.f && acc > tt) {
                    found = i;
                    break;
                }
            }
            s.bi[1] = found >= 0 ? found : lastpos;
        }
    }
    __syncthreads();
    *W_out = s.bf[0];
    const int r = s.bi[1];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(NT, 1) mentor_kernel(const __grid_constant__ MentorParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SharedM& s = *reinterpret_cast<SharedM*>(smem_raw);
    float* coarse = reinterpret_cast<float*>(smem_raw + ((sizeof(SharedM) + 15) & ~size_t(15)));
    const int tid = threadIdx.x;
    const int V = p.V, G1 = p.gamma + 1;
    const int ntask = p.B * p.gamma;
    const size_t slot = blockIdx.x;
    uint32_t* k0 = p.keys + slot * 2 * (size_t)V;
    uint32_t* k1 = k0 + V;
    uint32_t* i0 = p.idx + slot * 2 * (size_t)V;
    uint32_t* i1 = i0 + V;
    float* A = p.arr + slot * 7 * (size_t)V;
    const int nc = (V + kCoarse - 1) / kCoarse;

    for (int t = blockIdx.x; t < ntask; t += gridDim.x) {
        const int b = t / p.gamma, k = t - b * p.gamma;
        const TaskRec* rp = p.recs + (size_t)b * G1 + k;
        const int flags = rp->flags;
        int mflag = 0, mtok = -1;
        float alpha = -1.f, beta = 0.f;
        if ((flags & (kRecEData | kRecTimeout)) == 0 && !(flags & kRecAccept)) {
            Row r;
            r.c2 = p.c2;
            r.inv_t = p.inv_t;
            r.mtc = rp->m_t * p.c2;
            r.mdc = rp->m_d * p.c2;
            r.iSt = 1.f / rp->s_t;
            r.iSd = 1.f / rp->s_d;
            r.lnr0 = -(rp->m_t - rp->m_d) * p.inv_t - logf(rp->s_t) + logf(rp->s_d);
            r.bf16 = p.bf16;
            const size_t es = p.bf16 ? 2 : 4;
            r.rt = reinterpret_cast<const char*>(p.target) + ((size_t)b * G1 + k) * V * es;
            r.rd = reinterpret_cast<const char*>(p.draft) + ((size_t)b * p.gamma + k) * V * es;

            // KL(q || p) and the sort keys
            double kl0 = 0.0;
            {
                float acc = 0.f;
                for (int i = tid; i < V; i += NT) {
                    float q, pp, l;
                    qpl(r, i, q, pp, l);
                    acc += q * l;
                    k0[i] = f32_key(l);
                    i0[i] = (uint32_t)i;
                }
                kl0 = block_sum_d(s, (double)acc);
            }
            if (kl0 <= (double)p.kl_bound) {
                mflag = 1;
                alpha = 0.f;
            } else if (p.kl_bound == 0.f) {
                alpha = 1.f;
                beta = 1.f;
            } else {
                __threadfence_block();
                __syncthreads();
                radix_sort(s, k0, i0, k1, i1, V);
                // sorted arrays: L, CQ, CP, CL (prefix), SQ, SP (suffix), G
                float* L = A;
                float* CQ = A + V;
                float* CP = A + 2 * (size_t)V;
                float* CL = A + 3 * (size_t)V;
                float* SQ = A + 4 * (size_t)V;
                float* SP = A + 5 * (size_t)V;
                float* Gg = A + 6 * (size_t)V;
                const int per = (V + NT - 1) / NT;
                const int j0 = tid * per, j1 = min(V, j0 + per);
                float tq = 0.f, tp = 0.f, tl = 0.f;
                for (int j = j0; j < j1; ++j) {
                    float q, pp, l;
                    qpl(r, (int)__ldcg(i0 + j), q, pp, l);
                    L[j] = l;
                    tq += q;
                    tp += pp;
                    tl += q * l;
                }
                float eq = block_excl(s, tq), ep = block_excl(s, tp), el = block_excl(s, tl);
                for (int j = j0; j < j1; ++j) {
                    float q, pp, l;
                    qpl(r, (int)__ldcg(i0 + j), q, pp, l);
                    eq += q;
                    ep += pp;
                    el += q * l;
                    CQ[j] = eq;
                    CP[j] = ep;
                    CL[j] = el;
                }
                __syncthreads();
                {
                    // reverse order: thread NT-1-tid, chunk walked backwards
                    const int rt = NT - 1 - tid;
                    const int rj0 = rt * per, rj1 = min(V, rj0 + per);
                    float sq = 0.f, sp = 0.f;
                    for (int j = rj1 - 1; j >= rj0; --j) {
                        float q, pp, l;
                        qpl(r, (int)__ldcg(i0 + j), q, pp, l);
                        sq += q;
                        sp += pp;
                    }
                    float xq = block_excl(s, sq), xp = block_excl(s, sp);
                    for (int j = rj1 - 1; j >= rj0; --j) {
                        float q, pp, l;
                        qpl(r, (int)__ldcg(i0 + j), q, pp, l);
                        xq += q;
                        xp += pp;
                        SQ[j] = xq;
                        SP[j] = xp;
                        Gg[j] = xq * ex2(-l * 1.4426950408889634f) - xp;
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
                alpha = (float)hi;
                if (hi == 1.0) {
                    beta = 1.f;
                } else {
                    double bt;
                    if (tid == 0) {
                        kl_at(ar, hi, &bt);
                        s.bd[0] = bt;
                    }
                    __syncthreads();
                    beta = (float)s.bd[0];
                    __syncthreads();
                }
                s.bd[1] = hi;
            }
            if (alpha > 0.f) {
                // lossy test with the standard test's uniform
                const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
                const double rho = rp->p_x > 0.f ? (double)rp->q_x / (double)rp->p_x
                                                 : (rp->q_x > 0.f ? HUGE_VAL : 0.0);
                const double a = (alpha == 1.f) ? 1.0 : s.bd[1];
                mflag = (double)u < fmin(1.0, rho / a);
                if (!mflag) {
                    if (alpha == 1.f) {
                        mtok = rp->token;  // beta = 1: the standard residual draw
                    } else {
                        const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k,
                                                   kPurposeResample);
                        const float ib = 1.f / beta;
                        float W;
                        mtok = block_draw(s, V, u2, [&](int i) {
                            float q, pp, l;
                            qpl(r, i, q, pp, l);
                            return fmaxf(0.f, q * ib - pp);
                        }, &W);
                        if (!(W > 0.f))
                            mtok = block_draw(s, V, u2, [&](int i) {
                                float q, pp, l;
                                qpl(r, i, q, pp, l);
                                return q;
                            }, &W);
                    }
                }
            }
        } else if (flags & kRecAccept) {
            mflag = 1;
        }
        // record the position's decision; the last position of sequence b resolves it
        if (tid == 0) {
            p.m_flags[t] = mflag;
            p.m_token[t] = mtok;
            if (p.alpha_out) p.alpha_out[t] = (flags & kRecAccept) ? -1.f : alpha;
            if (p.beta_out) p.beta_out[t] = (flags & kRecAccept) ? 0.f : beta;
            __threadfence();
            const unsigned old = atomicAdd(&p.cnt[b], 1u);
            const int last = old == (unsigned)(p.gamma - 1);
            if (last) p.cnt[b] = 0u;
            s.bi[3] = last;
        }
        __syncthreads();
        if (s.bi[3]) {
            __threadfence();
            if (tid == 0) {
                int n = p.gamma, bad = 0;
                for (int i = 0; i < G1; ++i) bad |= p.recs[(size_t)b * G1 + i].flags & (kRecEData | kRecTimeout);
                for (int i = 0; i < p.gamma; ++i)
                    if (!__ldcg(p.m_flags + (size_t)b * p.gamma + i)) {
                        n = i;
                        break;
                    }
                const int tok = n < p.gamma ? __ldcg(p.m_token + (size_t)b * p.gamma + n)
                                            : p.recs[(size_t)b * G1 + p.gamma].token;
                const int st = (bad & kRecEData) ? kEData : (bad ? kETimeout : kOk);
                p.accepted[b] = st ? -1 : n;
                p.next_token[b] = st ? -1 : tok;
                if (p.status) p.status[b] = st;
                for (int j = 0; j < G1; ++j) {
                    int v = -1;
                    if (!st) v = j < n ? p.draft_tokens[(size_t)b * p.gamma + j] : (j == n ? tok : -1);
                    p.tokens[(size_t)b * G1 + j] = v;
                }
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

cudaError_t launch_mentor(const MentorParams& p, int grid, cudaStream_t stream) {
    const size_t smem = mentor_smem_bytes(p.V);
    cudaError_t e = cudaFuncSetAttribute(mentor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    mentor_kernel<<<grid, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sv
