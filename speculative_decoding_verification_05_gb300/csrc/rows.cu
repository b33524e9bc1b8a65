// Streaming row kernel: modified rejection sampling for temperature > 0.
//
// Work units are the logit rows of all sequences (2*gamma + 1 per sequence in
// verification: target rows k = 0..gamma, draft rows k = 0..gamma-1; P rows
// in sampling), each cut into `nseg` segments when rows are very long. CTAs
// take units from a global counter (dynamic scheduling, so a step of any
// shape balances over the SMs) and stream each unit once from HBM with
// 16-byte loads, keeping an online maximum and sum of exp2((z - m) log2e / T)
// per thread ("Accelerating Large Language Model Decoding with Speculative
// Sampling", "与标准采样方法的兼容性": the probabilities a transform acts on).
// The last segment of a row to finish turns the partial sums into the row's
// record (maximum, sum, top-k / top-p threshold and kept mass); the last row of
// a sequence to finish resolves the sequence (no thread ever waits for
// another CTA):
//
//   * acceptance left to right, u_k < min(1, q(x_k)/p(x_k)), stopping at the
//     first rejection n ("改进的拒绝采样");
//   * exactly one draw: from max(0, q_n - p_n) after a rejection, or the bonus
//     token from q_gamma when all gamma were accepted. The draw re-reads that
//     one row pair (fresh in L2) with the CTA-wide inverse CDF of draw.cuh.
//
// Top-p (fast path): while streaming, keys within kWin + 1 octaves of a
// CTA-wide running maximum are kept in shared memory; under the final maximum
// they contain every key whose mass is within 2^-kWin of the largest (an upper
// set in key order). A radix select over those keys with fixed-point masses
// (mass * 2^40, exact integers, so the result does not depend on summation
// order) gives tau, the largest key whose mass from the top reaches
// top_p * S, when the collected mass reaches that target. Top-k, rows whose
// crossing lies deeper and segmented rows take the exact slow path: the same
// radix select over the row read again from global memory, so both paths
// return the same tau and kept mass.

#include <algorithm>

#include "common.cuh"
#include "draw.cuh"

namespace sv {
namespace {

constexpr int NT = kDrawNT;
constexpr int NW = NT / 32;
constexpr int kMaxRows = 2 * 255 + 1;  // rows per sequence (verification, gamma <= 255)
constexpr int kWin = 13;               // fast top-p: keys within 2^-kWin of the row max
constexpr int kHeadCap = 4096;         // fast top-p: keys kept per row
constexpr float kFx = 1099511627776.0f;  // 2^40: masses >= 2^-17 are exact integers

struct Shared {
    int unit;
    int last;
    float red_m[NW], red_s[NW];
    unsigned long long ured[NW + 2];
    int bi[8];
    float bf[8];
    // fast top-p
    int nhead;
    unsigned hmax;                 // key of the CTA-wide running maximum
    uint32_t head[kHeadCap];
    unsigned long long hist[256];  // radix select
    // sequence resolve
    RowRec rec[kMaxRows];
    DrawShared draw;
};

SV_DEV float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Online (max, sum of exp2((z - max) c)) of one thread.
struct Online {
    float m;
    float s;
};

// Merge (bm, bs) into a (a.m becomes the larger maximum; NaN propagates).
SV_DEV void merge(Online& a, float bm, float bs, float c2) {
    if (!(bm <= a.m)) {  // b's maximum is larger, or NaN
        const float t = a.m;
        a.s = bs + (t == -INFINITY ? 0.f : a.s * ex2((t - bm) * c2));
        a.m = bm;
    } else if (bm != -INFINITY) {
        a.s += bs * ex2((bm - a.m) * c2);
    }
}

template <typename E>
struct Streamer {
    using T = VecTraits<E>;
    float c2;
    float wc;      // collection window in logits: (kWin + 1) / c2
    bool collect;  // top-p head collection
    Shared* s;

    SV_DEV void add_vec(Online& o, const float* x, int n, float hint) const {
        float vm = x[0];
#pragma unroll
        for (int e = 1; e < T::kN; ++e)
            if (e < n) vm = max_nan(vm, x[e]);
        if (!(vm <= o.m)) {
            o.s = (o.m == -INFINITY) ? 0.f : o.s * ex2((o.m - vm) * c2);
            o.m = vm;
        }
        if (o.m > -INFINITY || o.m != o.m) {
            const float mc = o.m * c2;
            const float cut = fmaxf(o.m, hint) - wc;
#pragma unroll
            for (int e = 0; e < T::kN; ++e) {
                if (e < n) {
                    o.s += ex2(fmaf(x[e], c2, -mc));
                    if (collect && x[e] > cut) {
                        const int slot = atomicAdd(&s->nhead, 1);
                        if (slot < kHeadCap) s->head[slot] = f32_key(x[e]);
                    }
                }
            }
        }
    }

    SV_DEV float shared_max() const { return key_to_f32(*reinterpret_cast<volatile unsigned*>(&s->hmax)); }

    // Streams elements [i0, i1) of row; returns this thread's online state.
    // Every thread of the CTA must call it (one barrier seeds the hint).
    SV_DEV Online run(const E* row, int i0, int i1) const {
        constexpr int es = sizeof(E);
        constexpr int VE = T::kN;
        constexpr int U = 4;
        Online o{-INFINITY, 0.f};
        const int tid = threadIdx.x;
        const uintptr_t a = (uintptr_t)(row + i0);
        const int head = min(i1 - i0, (int)(((16 - (a & 15)) & 15) / es));
        const int base = i0 + head;
        const int nb = (i1 - base) / VE;
        const uint4* vp = reinterpret_cast<const uint4*>(row + base);
        // first group of vectors; its maximum seeds the collection hint
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (tid + u * NT < nb) v[u] = ld_stream_v4(vp + tid + u * NT);
        float hint = -INFINITY;
        if (collect) {
            float vm = -INFINITY;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (tid + u * NT < nb) {
                    float x[VE];
                    T::unpack(v[u], x);
#pragma unroll
                    for (int e = 0; e < VE; ++e) vm = fmaxf(vm, x[e]);
                }
            }
            for (int o2 = 16; o2; o2 >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, o2));
            if ((tid & 31) == 0 && vm > -INFINITY) atomicMax(&s->hmax, f32_key(vm));
            __syncthreads();
            hint = shared_max();
        }
        if (tid < head) {
            float x[VE];
            x[0] = T::load1(row + i0 + tid);
            add_vec(o, x, 1, hint);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (tid + u * NT < nb) {
                float x[VE];
                T::unpack(v[u], x);
                add_vec(o, x, VE, hint);
            }
        }
        for (int j = tid + NT * U; j < nb; j += NT * U) {
            if (collect) {
                if (o.m > hint) atomicMax(&s->hmax, f32_key(o.m));
                hint = fmaxf(hint, shared_max());
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j + u * NT < nb) v[u] = ld_stream_v4(vp + j + u * NT);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j + u * NT < nb) {
                    float x[VE];
                    T::unpack(v[u], x);
                    add_vec(o, x, VE, hint);
                }
            }
        }
        const int t = base + nb * VE + tid;
        if (t < i1) {
            float x[VE];
            x[0] = T::load1(row + t);
            add_vec(o, x, 1, hint);
        }
        return o;
    }
};

// Block-wide merge of the threads' online states; the result in every thread.
// The tree order is fixed, so the result does not depend on timing.
SV_DEV Online block_merge(Shared& s, Online o, float c2) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float bm = __shfl_xor_sync(0xFFFFFFFFu, o.m, d);
        const float bs = __shfl_xor_sync(0xFFFFFFFFu, o.s, d);
        // the lower lane's state absorbs the higher lane's, in both lanes
        Online lo = (lane & d) ? Online{bm, bs} : o;
        const float hm = (lane & d) ? o.m : bm, hs = (lane & d) ? o.s : bs;
        merge(lo, hm, hs, c2);
        o = lo;
    }
    if (lane == 0) {
        s.red_m[warp] = o.m;
        s.red_s[warp] = o.s;
    }
    __syncthreads();
    Online r{s.red_m[0], s.red_s[0]};
    for (int w = 1; w < NW; ++w) merge(r, s.red_m[w], s.red_s[w], c2);
    __syncthreads();
    return r;
}

// Row r of sequence b.
template <typename E>
struct RowRef {
    const E* ptr;
    int k;       // draft position of the row
    bool has_x;  // the row takes part in an acceptance test (k < gamma)
};

template <typename E>
SV_DEV RowRef<E> row_ref(const RowParams& p, int b, int r) {
    RowRef<E> rr;
    if (p.mode == kModeSample) {
        rr.ptr = reinterpret_cast<const E*>(p.target) + ((size_t)b * p.rows_per_b + r) * p.V;
        rr.k = r;
        rr.has_x = false;
    } else if (r <= p.gamma) {
        rr.ptr = reinterpret_cast<const E*>(p.target) + ((size_t)b * (p.gamma + 1) + r) * p.V;
        rr.k = r;
        rr.has_x = r < p.gamma;
    } else {
        rr.k = r - p.gamma - 1;
        rr.ptr = reinterpret_cast<const E*>(p.draft) + ((size_t)b * p.gamma + rr.k) * p.V;
        rr.has_x = true;
    }
    return rr;
}

// --- exact thresholds ------------------------------------------------------

SV_DEV unsigned long long fx_mass(float z, float c2, float mc) {
    return __float2ull_rz(ex2(fmaf(z, c2, -mc)) * kFx);
}

// The top-p target top_p * (kept mass) in fixed point; both paths use it.
SV_DEV unsigned long long top_p_target(float top_p, unsigned long long kept) {
    return (unsigned long long)(top_p * (float)kept);
}

// Radix selection (8-bit digits, exact integer histograms) over n items given
// by src(i, key, w) -> valid: the largest key tau with W(key >= tau) >= target
// (W the sum of the valid items' w). Returns whether the valid items' total
// reaches the target; with *tau_out and *w_out = W(key >= tau) when it does,
// else the smallest key present and the total. Every thread returns the same.
// npass = 2 suffices for keys of bf16 values (their low 16 bits are fixed by
// the sign).
template <typename Src>
SV_DEV bool radix_select(Shared& s, const Src& src, int n, int npass, unsigned long long target,
                         uint32_t* tau_out, unsigned long long* w_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0;
    unsigned long long A = 0ull, wsel = 0ull;
    bool reach = true;
    for (int pass = 0; pass < npass; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += NT) s.hist[i] = 0ull;
        __syncthreads();
        for (int i = tid; i < n; i += NT) {
            uint32_t key;
            unsigned long long w;
            if (src(i, key, w) && (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8))))
                atomicAdd(&s.hist[(key >> shift) & 255u], w);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255 - 8l .. 248 - 8l (descending)
            unsigned long long h[8], L = 0ull;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                h[t] = s.hist[255 - 8 * lane - t];
                L += h[t];
            }
            unsigned long long P = L;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, P, d);
                if (lane >= d) P += y;
            }
            const unsigned long long total = __shfl_sync(0xFFFFFFFFu, P, 31);
            const bool ok = A + total >= target;
            unsigned long long cum = A + (P - L), above = 0ull;
            int dl = -1;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (ok) {
                    if (dl < 0 && h[t] > 0ull && cum + h[t] >= target) {
                        dl = t;
                        above = cum;
                    }
                } else if (h[t] > 0ull) {  // the lowest non-empty bin
                    dl = t;
                    above = cum;
                }
                cum += h[t];
            }
            const unsigned m = __ballot_sync(0xFFFFFFFFu, dl >= 0);
            const int src_lane = m ? (ok ? __ffs(m) - 1 : 31 - __clz(m)) : 0;
            if (lane == src_lane) {
                s.bi[1] = dl >= 0 ? 255 - 8 * lane - dl : 0;
                s.ured[NW] = dl >= 0 ? above : A;
                s.ured[NW + 1] = dl >= 0 ? above + h[dl] : A;
                s.bi[2] = ok;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)s.bi[1] << shift;
        A = s.ured[NW];
        wsel = s.ured[NW + 1];
        if (pass == 0) reach = s.bi[2] != 0;
        __syncthreads();
    }
    if (npass == 2) prefix |= (prefix & 0x80000000u) ? 0u : 0xFFFFu;
    *tau_out = prefix;
    *w_out = wsel;
    return reach;
}

// Fast top-p from the collected keys; false if the list overflowed or the
// crossing lies below the collected keys. Every thread returns the same value.
SV_DEV bool fast_top_p(Shared& s, const RowParams& p, float m, float S, int npass, float* thr, float* sk) {
    const int nh = s.nhead;
    if (nh > kHeadCap) return false;
    const float mc = m * p.c2, c2 = p.c2;
    const unsigned long long target = top_p_target(p.top_p, (unsigned long long)(S * kFx));
    const uint32_t* head = s.head;
    auto src = [&](int i, uint32_t& key, unsigned long long& w) {
        key = head[i];
        const float a = fmaf(key_to_f32(key), c2, -mc);
        w = __float2ull_rz(ex2(a) * kFx);
        return a > -(float)kWin;
    };
    uint32_t tau;
    unsigned long long kept;
    if (!radix_select(s, src, nh, npass, target, &tau, &kept)) return false;
    *thr = key_to_f32(tau);
    *sk = (float)kept * (1.0f / kFx);
    return true;
}

// Exact top-k / top-p over the row read from global memory (slow path).
template <typename E>
SV_DEV void slow_threshold(Shared& s, const RowParams& p, const E* row, float m, float S, float* thr,
                           float* sk) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float mc = m * p.c2, c2 = p.c2;
    constexpr int npass = sizeof(E) == 4 ? 4 : 2;
    uint32_t floor_key = 0u;
    unsigned long long kept = (unsigned long long)(S * kFx);
    float t = -INFINITY;
    if (p.transform & kXfTopK) {
        auto cnt = [&](int i, uint32_t& key, unsigned long long& w) {
            key = f32_key(VecTraits<E>::load1(row + i));
            w = 1ull;
            return true;
        };
        uint32_t kk;
        unsigned long long c;
        radix_select(s, cnt, p.V, npass, (unsigned long long)p.top_k, &kk, &c);
        floor_key = kk;
        t = key_to_f32(kk);
        unsigned long long part = 0ull;
        for (int i = tid; i < p.V; i += NT) {
            const float z = VecTraits<E>::load1(row + i);
            if (f32_key(z) >= kk) part += fx_mass(z, c2, mc);
        }
        for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
        if (lane == 0) s.ured[warp] = part;
        __syncthreads();
        kept = 0ull;
        for (int w = 0; w < NW; ++w) kept += s.ured[w];
        __syncthreads();
    }
    if (p.transform & kXfTopP) {
        auto mass = [&](int i, uint32_t& key, unsigned long long& w) {
            const float z = VecTraits<E>::load1(row + i);
            key = f32_key(z);
            w = fx_mass(z, c2, mc);
            return key >= floor_key;
        };
        uint32_t pk;
        unsigned long long w;
        radix_select(s, mass, p.V, npass, top_p_target(p.top_p, kept), &pk, &w);
        t = key_to_f32(pk);
        kept = w;
    }
    *thr = t;
    *sk = (float)kept * (1.0f / kFx);
}

// --- per-row draw (sampling) and per-sequence resolve (verification) --------

// One draw per row from its transformed probabilities, straight after the
// row's statistics (the row is still in L2).
template <typename E>
__device__ __noinline__ void sample_row(Shared& s, const RowParams& p, const E* row, int b, int r, int rowid) {
    const RowRec rec = s.rec[0];
    int tok = -1;
    if (!(rec.flags & kRecEData)) {
        const float u = uniform01(p.seed, p.offset + (uint64_t)b, p.pos0 + (uint32_t)r, p.purpose);
        tok = draw_q<E>(s.draw, row, p.V, rec, p.c2, u);
    }
    if (threadIdx.x == 0) {
        p.sample_out[rowid] = tok;
        if (tok < 0 && p.status) atomicMax(&p.status[b], kEData);
    }
}

// Sequence b, once all its rows have records: acceptance left to right up to
// the first rejection n, then exactly one draw (the residual of position n,
// or the bonus token from q_gamma), then the outputs.
template <typename E>
__device__ __noinline__ void resolve_sequence(Shared& s, const RowParams& p, int b) {
    const int tid = threadIdx.x;
    const int R = p.rows_per_b, G = p.gamma;
    __threadfence();
    for (int i = tid; i < R; i += NT) s.rec[i] = load_rec(p.rows + (size_t)b * R + i);
    __syncthreads();
    if (tid == 0) {
        int flags = 0;
        for (int i = 0; i < R; ++i) flags |= s.rec[i].flags;
        int n = G;
        for (int k = 0; k < G; ++k) {
            const RowRec& t = s.rec[k];
            const RowRec& d = s.rec[G + 1 + k];
            const float q = KeptExp{t.thr, p.c2, t.m * p.c2, 1.f}(t.zx) / t.Sk;
            const float pd = KeptExp{d.thr, p.c2, d.m * p.c2, 1.f}(d.zx) / d.Sk;
            if (p.probs_dbg) {
                p.probs_dbg[((size_t)b * G + k) * 2 + 0] = q;
                p.probs_dbg[((size_t)b * G + k) * 2 + 1] = pd;
            }
            if (n == G) {
                const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
                if (!accept_test(u, q, pd)) n = k;
            }
        }
        s.bi[2] = n;
        s.bi[3] = (flags & kRecEData) ? kEData : kOk;
    }
    __syncthreads();
    const int n = s.bi[2], stt = s.bi[3];
    int tok = -1;
    if (!stt) {
        const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)n, kPurposeResample);
        const RowRef<E> tr = row_ref<E>(p, b, n);
        if (n < G) {
            const RowRef<E> dr = row_ref<E>(p, b, G + 1 + n);
            tok = draw_residual<E>(s.draw, tr.ptr, dr.ptr, p.V, s.rec[n], s.rec[G + 1 + n], p.c2, u2);
        } else {
            tok = draw_q<E>(s.draw, tr.ptr, p.V, s.rec[G], p.c2, u2);
        }
    }
    if (tid == 0) {
        p.accepted[b] = stt ? -1 : n;
        p.next_token[b] = stt ? -1 : tok;
        if (p.status) p.status[b] = stt;
    }
    for (int j = tid; j <= G; j += NT) {
        int v = -1;
        if (!stt) v = j < n ? s.rec[j].x : (j == n ? tok : -1);
        p.tokens[(size_t)b * (G + 1) + j] = v;
    }
}

// --- the kernel -----------------------------------------------------------------

template <typename E, bool XF>
__global__ void __launch_bounds__(NT, 4) row_kernel(const __grid_constant__ RowParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Shared& s = *reinterpret_cast<Shared*>(smem_raw);
    const int tid = threadIdx.x;
    const int R = p.rows_per_b;
    const int nunits = p.B * R * p.nseg;
    const bool fast_p = XF && p.transform == kXfTopP && p.nseg == 1;
    const Streamer<E> st{p.c2, (float)(kWin + 1) / p.c2, fast_p, &s};

    for (;;) {
        if (tid == 0) {
            s.unit = (int)atomicAdd(p.work, 1u);
            s.nhead = 0;
            s.hmax = kKeyNegInf;
        }
        __syncthreads();
        const int unit = s.unit;
        if (unit >= nunits) break;
        const int rowid = unit / p.nseg, seg = unit - rowid * p.nseg;
        const int b = rowid / R, r = rowid - b * R;
        const RowRef<E> rr = row_ref<E>(p, b, r);
        const int i0 = seg * p.seg_len, i1 = min(p.V, i0 + p.seg_len);
        // the draft token and its logit in this row (loaded early, used at the end)
        int x = -1;
        float zx = 0.f;
        if (tid == 0 && rr.has_x) {
            x = p.draft_tokens[(size_t)b * p.gamma + rr.k];
            if (x >= i0 && x < i1) zx = VecTraits<E>::load1(rr.ptr + x);
        }

        const Online o = block_merge(s, st.run(rr.ptr, i0, i1), p.c2);

        // ---- row record (by the last segment of the row to finish) ----
        bool have_row = p.nseg == 1;
        float m = o.m, S = o.s;
        if (p.nseg > 1) {
            if (tid == 0) {
                SegRec sr;
                sr.m = o.m;
                sr.s = o.s;
                sr.zx = zx;
                sr.flags = 0;
                p.segs[unit] = sr;
                __threadfence();
                const unsigned old = atomicAdd(&p.row_cnt[rowid], 1u);
                s.last = old == (unsigned)(p.nseg - 1);
                if (s.last) p.row_cnt[rowid] = 0u;
            }
            __syncthreads();
            have_row = s.last != 0;
            if (have_row) {
                __threadfence();
                if (tid == 0) {
                    Online t{-INFINITY, 0.f};
                    for (int q = 0; q < p.nseg; ++q) {
                        const SegRec* sp = p.segs + (size_t)rowid * p.nseg + q;
                        merge(t, __ldcg(&sp->m), __ldcg(&sp->s), p.c2);
                        if (rr.has_x && x >= q * p.seg_len && x < (q + 1) * p.seg_len) zx = __ldcg(&sp->zx);
                    }
                    s.bf[0] = t.m;
                    s.bf[1] = t.s;
                }
                __syncthreads();
                m = s.bf[0];
                S = s.bf[1];
            }
        }
        if (have_row) {
            const bool bad = !(S > 0.f && S <= 3.0e38f);
            float thr = -INFINITY, sk = S;
            if (XF && !bad) {
                bool done = false;
                if (fast_p) done = fast_top_p(s, p, m, S, sizeof(E) == 4 ? 4 : 2, &thr, &sk);
                if (!done) slow_threshold<E>(s, p, rr.ptr, m, S, &thr, &sk);
            }
            if (tid == 0) {
                RowRec rec;
                rec.m = m;
                rec.S = S;
                rec.thr = thr;
                rec.Sk = sk;
                rec.zx = zx;
                rec.x = x;
                rec.flags = (bad || (rr.has_x && (x < 0 || x >= p.V))) ? kRecEData : 0;
                p.rows[rowid] = rec;
                s.rec[0] = rec;
            }
            __syncthreads();

            if (p.mode == kModeSample) {
                sample_row<E>(s, p, rr.ptr, b, r, rowid);
            } else if (p.mode == kModeVerify) {
                if (tid == 0) {
                    __threadfence();
                    const unsigned old = atomicAdd(&p.seq_cnt[b], 1u);
                    s.last = old == (unsigned)(R - 1);
                    if (s.last) p.seq_cnt[b] = 0u;
                }
                __syncthreads();
                if (s.last) resolve_sequence<E>(s, p, b);
            }
        }
        __syncthreads();
    }
}

template <typename E, bool XF>
cudaError_t launch_t(const RowParams& p, int sms, cudaStream_t stream) {
    auto kern = row_kernel<E, XF>;
    const size_t smem = sizeof(Shared);
    static const int per_sm = [&] {
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, smem) != cudaSuccess || n < 1)
            n = 1;
        return n;
    }();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.B * p.rows_per_b * p.nseg;
    const int grid = (int)std::min<long long>(units, (long long)sms * per_sm);
    kern<<<grid, NT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rows(const RowParams& p, int dtype, int sms, cudaStream_t stream) {
    const bool xf = p.transform != 0;
    if (dtype == 0) return xf ? launch_t<float, true>(p, sms, stream) : launch_t<float, false>(p, sms, stream);
    return xf ? launch_t<bf16_t, true>(p, sms, stream) : launch_t<bf16_t, false>(p, sms, stream);
}

}  // namespace sv
