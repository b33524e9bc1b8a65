// Inverse-CDF draw over one logit row (or a target/draft row pair) read from
// global memory by one CTA: the smallest index i with C_i > u W, where C is the
// inclusive prefix sum of the weights in index order and W their total; if
// rounding leaves no such index, the last index with positive weight.
//
// This is the draw behind the resampling step x ~ (q - p)+ and the bonus
// token of "Accelerating Large Language Model Decoding with Speculative
// Sampling" ("改进的拒绝采样"), and behind the mentor variant's
// s ~ max(0, q/beta - p). Every caller uses this one routine, so equal inputs
// give bit-identical tokens on every path.
//
// The row is cut into rounds of NT * PER consecutive elements; inside a round
// thread t owns PER consecutive elements. Pass 1 sums every round with a fixed
// order (thread: left to right; warp: a butterfly over the lanes) and keeps
// the per-warp totals; warp 0 adds the rounds in a fixed order (lane l owns
// consecutive rounds) and finds the crossing round; pass 2 re-reads only that
// round and walks warps, lanes and elements down to the token.
#pragma once

#include "common.cuh"

namespace sv {

constexpr int kDrawNT = 256;
constexpr int kDrawNW = kDrawNT / 32;
constexpr int kDrawMaxRounds = 128;  // covers V <= SPEC_MAX_V for every element size
// Vectors per row, thread and round in the kernels that only draw: four for
// fp32 rows (long rows, fewer rounds), two for bf16 (shorter rows, fewer
// registers). The verification draw and the mentor resolve use the same.
template <typename E>
constexpr int draw_vec() { return sizeof(E) == 4 ? 4 : 2; }

struct DrawShared {
    float wt[kDrawMaxRounds][kDrawNW];  // per-round, per-warp totals
    float W;
    int round;
    float rem;
    int token;
};

// Elements per thread per round (kVec 16-byte vectors).
template <typename E, int kVec = 2>
constexpr int draw_per() { return kVec * (16 / (int)sizeof(E)); }

// Loads the PER logits of (row, i0 .. i0 + PER) as fp32 (-inf beyond V).
template <typename E, int kVec = 2>
SV_DEV void draw_load(const E* row, int i0, int V, float (&x)[draw_per<E, kVec>()]) {
    constexpr int PER = draw_per<E, kVec>();
    constexpr int VE = 16 / (int)sizeof(E);
    const uintptr_t a = (uintptr_t)(row + i0);
    if (i0 + PER <= V && (a & 15) == 0) {
#pragma unroll
        for (int h = 0; h < kVec; ++h) {
            const uint4 r = __ldg(reinterpret_cast<const uint4*>(row + i0) + h);
            float y[VE];
            VecTraits<E>::unpack(r, y);
#pragma unroll
            for (int e = 0; e < VE; ++e) x[h * VE + e] = y[e];
        }
    } else {
#pragma unroll
        for (int e = 0; e < PER; ++e)
            x[e] = (i0 + e < V) ? VecTraits<E>::load1(row + i0 + e) : -INFINITY;
    }
}

// Draw with weights wf(zt, zd) of the target row rt and (optional) draft row
// rd. Returns the token (same value in every thread); *W_out the total.
// All threads of the CTA must call it; a CTA wider than kDrawNT threads works
// with its first kDrawNT threads (the others only join the barriers), so the
// summation order and the result do not depend on the caller's CTA size.
// kVec: 16-byte vectors of each row per thread and round. 4 (the kernels that
// only draw) keeps more loads in flight; 2 (draws inside the streaming
// kernel) needs fewer registers. Equal kVec gives bit-identical results.
template <typename E, typename WF, int kVec = 2>
SV_DEV int block_draw(DrawShared& ds, const E* rt, const E* rd, int V, float u, WF wf, float* W_out) {
    constexpr int PER = draw_per<E, kVec>();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool act = tid < kDrawNT;
    const int rounds = (V + kDrawNT * PER - 1) / (kDrawNT * PER);
    auto thread_sum = [&](int r, float (&w)[PER]) {
        const int i0 = r * kDrawNT * PER + tid * PER;
        float xt[PER], xd[PER];
        draw_load<E, kVec>(rt, i0, V, xt);
        if (rd) draw_load<E, kVec>(rd, i0, V, xd);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            w[e] = (i0 + e < V) ? wf(xt[e], rd ? xd[e] : -INFINITY) : 0.f;
            acc += w[e];
        }
        return acc;
    };
    // pass 1: per-round, per-warp totals
    for (int r = 0; act && r < rounds; ++r) {
        float wsum;
        if constexpr (kVec == 2) {
            float w[PER];
            wsum = thread_sum(r, w);
        } else {
            // as thread_sum (same elements, same order) from the raw vectors,
            // all kVec vectors of both rows in flight, the weights not kept
            constexpr int VE = 16 / (int)sizeof(E);
            const int i0 = r * kDrawNT * PER + tid * PER;
            const uintptr_t at = (uintptr_t)(rt + i0), ad = rd ? (uintptr_t)(rd + i0) : 0;
            if (i0 + PER <= V && ((at | ad) & 15) == 0) {
                uint4 vt[kVec], vd[kVec];
#pragma unroll
                for (int h = 0; h < kVec; ++h) {
                    vt[h] = __ldg(reinterpret_cast<const uint4*>(rt + i0) + h);
                    if (rd) vd[h] = __ldg(reinterpret_cast<const uint4*>(rd + i0) + h);
                }
                wsum = 0.f;
#pragma unroll
                for (int h = 0; h < kVec; ++h) {
                    float yt[VE], yd[VE];
                    VecTraits<E>::unpack(vt[h], yt);
                    if (rd) VecTraits<E>::unpack(vd[h], yd);
#pragma unroll
                    for (int e = 0; e < VE; ++e) wsum += wf(yt[e], rd ? yd[e] : -INFINITY);
                }
            } else {
                float w[PER];
                wsum = thread_sum(r, w);
            }
        }
        // butterfly: every lane ends with the same warp total, in a fixed order
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, o);
        if (lane == 0 && SV_IN(r, kDrawMaxRounds)) ds.wt[r][warp] = wsum;
    }
    __syncthreads();
    if (warp == 0) {
        // round totals in a fixed order; lane l owns rounds [l * per, (l + 1) * per)
        const int per = (rounds + 31) / 32;
        const int q0 = min(rounds, lane * per), q1 = min(rounds, q0 + per);
        float lsum = 0.f;
        for (int r = q0; r < q1; ++r) {
            float R = 0.f;
            for (int w = 0; w < kDrawNW; ++w) R += ds.wt[r][w];
            lsum += R;
        }
        float W;
        const float lpre = warp_seq_exclusive(lsum, &W);
        const float t = u * W;
        // the round holding the crossing: the last round whose start <= t with positive weight
        float carry = lpre, rem = 0.f;
        int rr = -1;
        for (int r = q0; r < q1; ++r) {
            float R = 0.f;
            for (int w = 0; w < kDrawNW; ++w) R += ds.wt[r][w];
            if (carry <= t && R > 0.f) {
                rr = r;
                rem = t - carry;
            }
            carry += R;
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, rr >= 0);
        if (lane == (m ? 31 - __clz(m) : 0)) {
            ds.W = W;
            ds.round = rr;
            ds.rem = rem;
            ds.token = -1;
        }
    }
    __syncthreads();
    const int rr = ds.round;
    *W_out = ds.W;
    if (act && rr >= 0) {
        // pass 2: the crossing round only
        float w[PER];
        const float tsum = thread_sum(rr, w);
        float wtot;
        const float lane_pre = warp_seq_exclusive(tsum, &wtot);
        const float rem = ds.rem;
        int ow = -1;
        float wpre = 0.f, acc = 0.f;
        for (int q = 0; q < kDrawNW; ++q) {
            if (acc <= rem && ds.wt[rr][q] > 0.f) {
                ow = q;
                wpre = acc;
            }
            acc += ds.wt[rr][q];
        }
        if (warp == ow) {
            const float tw = rem - wpre;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, lane_pre <= tw && tsum > 0.f);
            const int ol = m ? 31 - __clz(m) : -1;
            if (lane == ol) {
                const float tt = tw - lane_pre;
                const int i0 = rr * kDrawNT * PER + tid * PER;
                float c = 0.f;
                int found = -1, lastpos = -1;
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    if (w[e] > 0.f) lastpos = i0 + e;
                    c += w[e];
                    if (found < 0 && w[e] > 0.f && c > tt) found = i0 + e;
                }
                ds.token = found >= 0 ? found : lastpos;
            }
        }
    }
    __syncthreads();
    const int tok = ds.token;
    __syncthreads();
    return tok;
}

// exp2((z - m) log2e / T) for a kept logit (z >= thr), times `scale`; 0 otherwise.
struct KeptExp {
    float thr, c2, mc, scale;
    SV_DEV float operator()(float z) const { return z >= thr ? ex2(fmaf(z, c2, -mc)) * scale : 0.f; }
};

// Residual weight max(0, q_i - p_i) of a target/draft row pair.
struct ResidualW {
    KeptExp q, p;
    SV_DEV float operator()(float zt, float zd) const { return fmaxf(0.f, q(zt) - p(zd)); }
};

// max(0, q - l p) with l the lenience (1: the exact residual (q - p)+).
SV_DEV ResidualW residual_weight(const RowRec& t, const RowRec& d, float c2, float l = 1.f) {
    return ResidualW{KeptExp{t.thr, c2, t.m * c2, 1.f / t.Sk}, KeptExp{d.thr, c2, d.m * c2, l * (1.f / d.Sk)}};
}

// Accept with probability min(1, q/p): u < q/p; p = 0 accepts iff q > 0.
SV_DEV bool accept_test(float u, float q, float p) {
    const float ratio = p > 0.f ? q / p : (q > 0.f ? INFINITY : 0.f);
    return u < ratio;
}

// Inverse-CDF draw from the (transformed) row's probabilities q (sampling and
// the bonus token).
template <typename E, int kVec = 2>
SV_DEV int draw_q(DrawShared& ds, const E* row, int V, const RowRec& r, float c2, float u) {
    const KeptExp q{r.thr, c2, r.m * c2, 1.f};
    float W;
    auto wq = [&](float zt, float) { return q(zt); };
    return block_draw<E, decltype(wq), kVec>(ds, row, (const E*)nullptr, V, u, wq, &W);
}

// Residual draw x ~ max(0, q - l p) over a target/draft row pair (l = 1: the
// exact residual); from q when the residual vanishes (q = l p to rounding).
template <typename E, int kVec = 2>
SV_DEV int draw_residual(DrawShared& ds, const E* rt, const E* rd, int V, const RowRec& t, const RowRec& d,
                         float c2, float u, float l = 1.f) {
    const ResidualW w = residual_weight(t, d, c2, l);
    float W;
    const int tok = block_draw<E, ResidualW, kVec>(ds, rt, rd, V, u, w, &W);
    if (W > 0.f) return tok;
    return draw_q<E, kVec>(ds, rt, V, t, c2, u);
}

// Records are 32 bytes on 16-byte boundaries of the workspace: two 16-byte
// loads (cached in L2 only: records written earlier in the same kernel).
static_assert(sizeof(RowRec) == 32, "row records are two 16-byte words");
SV_DEV RowRec load_rec(const RowRec* src) {
    const uint4 a = __ldcg(reinterpret_cast<const uint4*>(src));
    const uint4 b = __ldcg(reinterpret_cast<const uint4*>(src) + 1);
    RowRec q;
    q.m = __uint_as_float(a.x);
    q.S = __uint_as_float(a.y);
    q.thr = __uint_as_float(a.z);
    q.Sk = __uint_as_float(a.w);
    q.zx = __uint_as_float(b.x);
    q.x = (int32_t)b.y;
    q.flags = (int32_t)b.z;
    q.nkept = (int32_t)b.w;
    return q;
}

}  // namespace sv
