// Exact top-k / top-p thresholds over a set of logits, shared by the row
// kernels: the kept set of a row is {z >= tau}, tau the largest key whose
// weight from the top (a count for top-k; for top-p the fixed-point mass
// round_down(2^a 2^40), a = (z - m) log2e / T, summed as exact integers so
// that the result does not depend on summation order) reaches the target
// ("Accelerating Large Language Model Decoding with Speculative Sampling",
// "与标准采样方法的兼容性": the transforms act on the distributions the scheme
// samples from). Every function here is called by all kSelNT threads of a
// CTA; `each(f)` calls f(valid, key, a) once per item, the same number of
// times in every lane of a warp. The shared-state type SH provides
// h.g (GenSel), bi[8], ured[kSelNW + 2], nsel and odirty.
#pragma once

#include "common.cuh"

namespace sv {
namespace sel {

constexpr int kSelNT = 256;
constexpr int kSelNW = kSelNT / 32;
constexpr int kSel = 256;                // keys compared exactly inside the crossing bin
constexpr float kFx = 1099511627776.0f;  // 2^40: masses >= 2^-17 are exact integers

struct GenSel {
    unsigned hcnt[256];               // selection histogram: counts
    unsigned long long hist[256];     //                      fixed-point masses
    uint32_t skey[kSel];              // keys of the crossing bin
    unsigned long long smass[kSel];
};

SV_DEV float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

SV_DEV uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

SV_DEV float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
SV_DEV float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// --- exact thresholds ------------------------------------------------------

// round_toward_zero(2^a * 2^40) for a <= 0, from the bits of v = 2^a 2^40
// (exact in fp32: a power-of-two scaling of ex2's result): v = M 2^e with
// M the 24-bit significand, so floor(v) = M << e, or M >> -e below 2^23.
// Integer operations only (conversions share the MUFU pipe with ex2).
SV_DEV unsigned long long fx_of(float a) {
    const uint32_t b = __float_as_uint(ex2(a) * kFx);
    const int e = (int)(b >> 23) - 150;
    const uint32_t M = (b & 0x7FFFFFu) | 0x800000u;
    if (b < 0x00800000u || e <= -24 || b >= 0x7F800000u) return 0ull;  // below 1, zero, or not finite
    return e >= 0 ? (unsigned long long)M << e : (unsigned long long)(M >> -e);
}

// The top-p target top_p * (kept mass) in fixed point; both paths use it.
SV_DEV unsigned long long top_p_target(float top_p, unsigned long long kept) {
    const unsigned long long t = (unsigned long long)(top_p * (float)kept);
    return t ? t : 1ull;
}

// Bin of a = (z - m) log2e / T <= 0, non-increasing in z: 1/16 octave down to
// 12 octaves, then 1 octave down to 60, then 8 octaves down to 180, then the
// rest (and -inf).
SV_DEV int abin(float a) {
    const float t = -a;
    if (t < 12.f) return max(0, (int)(t * 16.f));
    if (t < 60.f) return 192 + (int)(t - 12.f);
    if (t < 180.f) return 240 + (int)((t - 60.f) * 0.125f);
    return 255;
}

template <typename SH>
SV_DEV unsigned long long block_sum_u64(SH& s, unsigned long long v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) s.ured[warp] = v;
    __syncthreads();
    unsigned long long t = 0ull;
    for (int w = 0; w < kSelNW; ++w) t += s.ured[w];
    __syncthreads();
    return t;
}

template <typename SH>
SV_DEV uint32_t block_max_u32(SH& s, uint32_t v) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (lane == 0) s.ured[warp] = v;
    __syncthreads();
    uint32_t t = 0u;
    for (int w = 0; w < kSelNW; ++w) t = max(t, (uint32_t)s.ured[w]);
    __syncthreads();
    return t;
}

// Histogram add with the lanes of a warp that hit the same bin combined into
// one atomic per bin. Every lane of the warp must call it (v: item valid).
// Histogram add, one shared atomic per valid lane: for items spread over many
// bins (the candidates near a row's maximum), where combining the lanes of a
// bin first (hist_add) costs a pass per distinct bin.
template <typename SH>
SV_DEV void hist_add_sparse(SH& s, bool v, int bin, unsigned long long w) {
    if (v) {
        atomicAdd(&s.h.g.hist[bin], w);
        atomicAdd(&s.h.g.hcnt[bin], 1u);
    }
}

template <typename SH>
SV_DEV void hist_add(SH& s, bool v, int bin, unsigned long long w) {
    const unsigned act = __ballot_sync(0xFFFFFFFFu, v);
    if (v) {
        const unsigned peers = __match_any_sync(act, bin);
        const unsigned lo = __reduce_add_sync(peers, (unsigned)(w & 0x1FFFFFull));
        const unsigned hi = __reduce_add_sync(peers, (unsigned)(w >> 21));  // w < 2^41
        if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) {
            atomicAdd(&s.h.g.hist[bin], ((unsigned long long)hi << 21) + lo);
            atomicAdd(&s.h.g.hcnt[bin], (unsigned)__popc(peers));
        }
    }
}

// SPARSE: items over many bins (one atomic per lane); else lanes of a bin combined.
template <bool SPARSE, typename SH>
SV_DEV void hist_put(SH& s, bool v, int bin, unsigned long long w) {
    if constexpr (SPARSE) hist_add_sparse(s, v, bin, w); else hist_add(s, v, bin, w);
}

struct Sel {
    uint32_t tau;                 // selected key
    unsigned long long cnt, mass; // count and fixed-point mass of the items with key >= tau
    bool reach;                   // the items' total reached the target
};

// Radix selection (8-bit digits, exact integer histograms) restricted to the
// items accepted by `keep`, starting above weight A0: the largest key tau with
// A0 + W(key >= tau) >= target. npass = 2 suffices for keys of bf16 values.
template <bool SPARSE, typename SH, typename Each, typename Keep>
SV_DEV uint32_t radix_select(SH& s, const Each& each, const Keep& keep, int npass, bool by_count,
                             unsigned long long A0, unsigned long long target) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t prefix = 0;
    unsigned long long A = A0;
    for (int pass = 0; pass < npass; ++pass) {
        const int shift = 24 - 8 * pass;
        if (threadIdx.x == 0) s.odirty = 1;
        for (int i = threadIdx.x; i < 256; i += kSelNT) {
            s.h.g.hist[i] = 0ull;
            s.h.g.hcnt[i] = 0u;
        }
        __syncthreads();
        each([&](bool v, uint32_t key, float a) {
            v = v && keep(key, a) && (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8)));
            hist_put<SPARSE>(s, v, v ? (int)((key >> shift) & 255u) : 0, v && !by_count ? fx_of(a) : 0ull);
        });
        __syncthreads();
        if (warp == 0) {
            // lane l owns digits 255 - 8l .. 248 - 8l (descending keys)
            unsigned long long h[8], L = 0ull;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int d = 255 - 8 * lane - t;
                h[t] = by_count ? (unsigned long long)s.h.g.hcnt[d] : s.h.g.hist[d];
                L += h[t];
            }
            unsigned long long P = L;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, P, d);
                if (lane >= d) P += y;
            }
            unsigned long long cum = A + (P - L), above = 0ull;
            int dl = -1, lastnz = -1;
            unsigned long long above_last = 0ull;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (dl < 0 && h[t] > 0ull && cum + h[t] >= target) {
                    dl = t;
                    above = cum;
                }
                if (h[t] > 0ull) {
                    lastnz = t;
                    above_last = cum;
                }
                cum += h[t];
            }
            const unsigned mf = __ballot_sync(0xFFFFFFFFu, dl >= 0);
            const unsigned ml = __ballot_sync(0xFFFFFFFFu, lastnz >= 0);
            // the crossing digit, else (target not reached) the lowest non-empty digit
            const int src = mf ? __ffs(mf) - 1 : (ml ? 31 - __clz(ml) : 0);
            if (lane == src) {
                const int t = mf ? dl : lastnz;
                s.bi[1] = t >= 0 ? 255 - 8 * lane - t : 0;
                s.ured[kSelNW] = t >= 0 ? (mf ? above : above_last) : A;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)s.bi[1] << shift;
        A = s.ured[kSelNW];
        __syncthreads();
    }
    if (npass == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    return prefix;
}

// Exact weighted selection over the items of `each` with key >= floor_key:
// tau = the largest key with W(key >= tau) >= target, W a count (by_count) or
// the fixed-point mass. Every thread returns the same result. Unreached
// targets return reach = false (tau and the sums are then unspecified).
template <bool SPARSE, typename SH, typename Each>
SV_DEV Sel select(SH& s, const Each& each, int npass, bool by_count, uint32_t floor_key,
                  unsigned long long target) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256; i += kSelNT) {
        s.h.g.hist[i] = 0ull;
        s.h.g.hcnt[i] = 0u;
    }
    if (tid == 0) {
        s.nsel = 0;
        s.odirty = 1;
    }
    __syncthreads();
    each([&](bool v, uint32_t key, float a) {
        v = v && key >= floor_key;
        hist_put<SPARSE>(s, v, v ? abin(a) : 0, v ? fx_of(a) : 0ull);
    });
    __syncthreads();
    if (warp == 0) {
        // lane l owns bins 8l .. 8l + 7 (descending keys)
        unsigned long long h[8], L = 0ull;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            h[t] = by_count ? (unsigned long long)s.h.g.hcnt[8 * lane + t] : s.h.g.hist[8 * lane + t];
            L += h[t];
        }
        unsigned long long P = L;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, P, d);
            if (lane >= d) P += y;
        }
        const bool reach = __shfl_sync(0xFFFFFFFFu, P, 31) >= target;
        unsigned long long cum = P - L;
        int dl = -1;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (dl < 0 && h[t] > 0ull && cum + h[t] >= target) dl = t;
            cum += h[t];
        }
        const unsigned mf = __ballot_sync(0xFFFFFFFFu, dl >= 0);
        const int c = mf ? 8 * (__ffs(mf) - 1) + __shfl_sync(0xFFFFFFFFu, dl, __ffs(mf) - 1) : 0;
        // weights of the bins above c: count, mass
        unsigned long long ac = 0ull, am = 0ull;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (8 * lane + t < c) {
                ac += s.h.g.hcnt[8 * lane + t];
                am += s.h.g.hist[8 * lane + t];
            }
        }
        for (int o = 16; o; o >>= 1) {
            ac += __shfl_xor_sync(0xFFFFFFFFu, ac, o);
            am += __shfl_xor_sync(0xFFFFFFFFu, am, o);
        }
        if (lane == 0) {
            s.bi[0] = reach && mf;
            s.bi[1] = c;
            s.ured[kSelNW] = ac;
            s.ured[kSelNW + 1] = am;
        }
    }
    __syncthreads();
    Sel r;
    r.reach = s.bi[0] != 0;
    const int c = s.bi[1];
    const unsigned long long ac = s.ured[kSelNW], am = s.ured[kSelNW + 1];
    const int nc = (int)s.h.g.hcnt[c];
    __syncthreads();
    if (!r.reach) return r;
    const unsigned long long above = by_count ? ac : am;
    if (nc <= kSel) {
        // the crossing bin's keys, compared exactly
        each([&](bool v, uint32_t key, float a) {
            if (v && key >= floor_key && abin(a) == c) {
                const int slot = atomicAdd(&s.nsel, 1);
                s.h.g.skey[slot] = key;
                s.h.g.smass[slot] = fx_of(a);
            }
        });
        __syncthreads();
        const int n = s.nsel;
        uint32_t cand = 0u;
        for (int i = tid; i < n; i += kSelNT) {
            const uint32_t ki = s.h.g.skey[i];
            unsigned long long W = above;
            for (int j = 0; j < n; ++j) W += s.h.g.skey[j] >= ki ? (by_count ? 1ull : s.h.g.smass[j]) : 0ull;
            if (W >= target) cand = max(cand, ki);
        }
        r.tau = block_max_u32(s, cand);
        unsigned long long pc = 0ull, pm = 0ull;
        for (int i = tid; i < n; i += kSelNT) {
            if (s.h.g.skey[i] >= r.tau) {
                pc += 1ull;
                pm += s.h.g.smass[i];
            }
        }
        r.cnt = ac + block_sum_u64(s, pc);
        r.mass = am + block_sum_u64(s, pm);
    } else {
        auto keep = [&](uint32_t key, float a) { return key >= floor_key && abin(a) == c; };
        r.tau = radix_select<SPARSE>(s, each, keep, npass, by_count, above, target);
        unsigned long long pc = 0ull, pm = 0ull;
        each([&](bool v, uint32_t key, float a) {
            if (v && key >= r.tau) {
                pc += 1ull;
                pm += fx_of(a);
            }
        });
        r.cnt = block_sum_u64(s, pc);
        r.mass = block_sum_u64(s, pm);
    }
    return r;
}

// Top-k then top-p over the items of `each`. Returns false (head keys only)
// when they do not decide the threshold; the row path always decides.
template <bool SPARSE, typename SH, typename Each>
SV_DEV bool threshold_from(SH& s, const RowParams& p, const Each& each, int npass, bool head, float S,
                           float* thr, float* sk) {
    unsigned long long kept = (unsigned long long)(S * kFx);
    float t = -INFINITY;
    uint32_t floor_key = 0u;
    if (p.transform & kXfTopK) {
        const Sel r = select<SPARSE>(s, each, npass, true, 0u, (unsigned long long)p.top_k);
        if (!r.reach) {
            if (head) return false;
        } else {
            floor_key = r.tau;
            t = key_to_f32(r.tau);
            kept = r.mass;
        }
    }
    if (p.transform & kXfTopP) {
        const Sel r = select<SPARSE>(s, each, npass, false, floor_key, top_p_target(p.top_p, kept));
        if (!r.reach) {
            if (head) return false;
        } else {
            t = key_to_f32(r.tau);
            kept = r.mass;
        }
    }
    *thr = t;
    *sk = (float)kept * (1.0f / kFx);
    return true;
}

// bf16 ordinal: order-preserving 16-bit key of a bf16 value (-0 folded onto +0).
SV_DEV uint32_t ord16(uint32_t raw) {
    raw = raw == 0x8000u ? 0u : raw;
    return (raw & 0x8000u) ? (~raw & 0xFFFFu) : (raw | 0x8000u);
}

SV_DEV float ord16_value(uint32_t k) {
    const uint32_t raw = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(raw << 16);
}

}  // namespace sel
}  // namespace sv
