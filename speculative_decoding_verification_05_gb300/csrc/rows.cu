// Streaming row kernel: modified rejection sampling for temperature > 0.
//
// Work units are the logit rows of all sequences (2*gamma + 1 per sequence in
// verification: target rows k = 0..gamma, draft rows k = 0..gamma-1; P rows
// in sampling), each cut into `nseg` segments when rows are long and few.
// CTAs take units from a global counter (dynamic scheduling, so a step of any
// shape balances over the SMs) and stream each unit once from HBM with
// 16-byte loads. Per row the CTA computes the maximum m and
// S = sum_i exp2((z_i - m) log2e / T), the normaliser of the probabilities a
// transform acts on ("Accelerating Large Language Model Decoding with
// Speculative Sampling", "与标准采样方法的兼容性"). The exponentials are taken
// against a fixed reference, the maximum of the first group of vectors the
// CTA loads (one block reduction), so the loop needs no running rescale; S is
// moved to m once at the end (a row whose sum overflows against the
// reference is summed again against m). The last segment of a row to finish
// writes the row's record (maximum, sum, top-k / top-p threshold and kept
// mass); the last row of a sequence to finish resolves the sequence (no
// thread ever waits for another CTA): acceptance left to right,
// u_k < min(1, q(x_k)/p(x_k)), stopping at the first rejection n
// ("改进的拒绝采样"), the accepted prefix, and n. The draw kernel then makes
// each sequence's one draw: from max(0, q_n - p_n) after a rejection, or the
// bonus token from q_gamma when all gamma were accepted, with the CTA-wide
// inverse CDF of draw.cuh over that one row pair. Five 256-thread CTAs run
// per SM.
//
// Thresholds (top-k, top-p). While streaming, each thread stores in its own
// shared-memory slots the logits above (reference - (kWin + 1) octaves) (fp32:
// the keys; bf16: the 32-bit word of each adjacent pair with a logit above);
// they form an upper set in key order that holds every logit whose mass is
// within 2^-kWin of the largest (bf16 rows: kWinB while streaming). A bf16
// row whose slots overflow is stored again from the row with the same window
// below its finished maximum; one whose stored keys still do not decide the
// threshold is stored again with kWinWide + 1 octaves below it;// again from L2 with the cut of its finished maximum. tau is the largest key whose weight from the top (a
// count for top-k, the fixed-point mass * 2^40 for top-p: exact integers, so
// independent of summation order) reaches the target. bf16 rows count the
// stored keys per distinct bf16 value (a histogram over the ordinals of the
// values just below the reference) and scan it once; fp32 rows use a
// histogram over a monotone function of the logit (1/16 octave bins near the
// maximum) and compare the keys of the crossing bin exactly. When the stored
// keys do not decide the threshold (a thread's slots overflowed, the crossing
// lies deeper, or the row is split into segments) the same selection runs
// over the row read again from global memory, so every path gives the same
// tau and kept mass.

#include <algorithm>

#include "common.cuh"
#include "draw.cuh"
#include "select.cuh"

namespace sv {
namespace {

using namespace sel;

constexpr int NT = kDrawNT;
constexpr int NW = NT / 32;
constexpr int kMaxRows = 2 * 255 + 1;  // rows per sequence (verification, gamma <= 255)
constexpr int kU = 4;                  // 16-byte vectors in flight per thread
constexpr int kWin = 13;               // stored keys: within 2^-kWin of the row max (plus one octave)
constexpr int kWinB = 11;              // bf16 rows while streaming (a second, wider pass if needed)
constexpr int kWinWide = 15;           // bf16 second pass: the ordinal histogram's reach
constexpr int kSlotBytes = 96;         // key slots per thread, in bytes (five CTAs per SM fit)
constexpr int kOrd = 2048;             // bf16 ordinal histogram: bins
constexpr uint32_t kPrefetchBytes = 65536;  // next units up to this size are prefetched into L2


struct Shared {
    int q[3];                         // work units: this one and the next two
    int last;
    unsigned hmax;                    // key of the first group's maximum
    int ovf;                          // a thread's key slots overflowed
    int nsel;
    float red_m[NW], red_s[NW];
    unsigned long long ured[NW + 2];
    unsigned long long ured2[NW];
    int bi[8];
    float bf[8];
    unsigned short hn[NT];            // stored keys (fp32) or key pairs (bf16) per thread
    float cut;                        // the row's storage cut
    union {
        GenSel g;                     // binned selection (fp32 rows, global fallback)
        unsigned ocnt[kOrd];          // bf16 rows: stored keys per distinct value
    } h;
    int jmax;                         // deepest ordinal bin in use
    int odirty;                       // h.g was used since h.ocnt was last cleared
    union {
        unsigned char slots[kSlotBytes * NT];  // slot c of thread t at element c * NT + t
        RowRec rec[kMaxRows];                  // sequence resolve (after the row's threshold)
    } u;
    DrawShared draw;
};


// Online (max, sum of exp2((z - max) c)) of a segment.
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

// --- streaming core ------------------------------------------------------------

// Stores the raw bits of logits above `cut` in the thread's slots.
template <typename K>
struct Collect {
    static constexpr int kPer = kSlotBytes / (int)sizeof(K);
    K* base;  // slot 0 of this thread; slot c at base[c * NT]
    float cut;
    int hc;
    SV_DEV void operator()(float x, uint32_t raw) {
        if (x > cut) {
            if (hc < kPer) base[hc * NT] = (K)raw;
            ++hc;
        }
    }
    // Branch-free form for when at least one slot is free: the key is always
    // written to the next slot and kept only if it passes the cut.
    SV_DEV void put(float x, uint32_t raw) {
        if (SV_IN(hc, kPer)) base[hc * NT] = (K)raw;
        hc += x > cut;
    }
};

// bf16 rows: the 32-bit word of two adjacent logits goes to the thread's
// slots when either of them is above `cut` (one store per pair); the reader
// checks both halves against the cut again.
struct PairCollect {
    static constexpr int kPer = kSlotBytes / 4;
    uint32_t* base;  // slot 0 of this thread; slot c at base[c * NT]
    float cut;
    int hc;
    // branch-free, for when a slot is free
    SV_DEV void put(float lo, float hi, uint32_t w) {
        if (SV_IN(hc, kPer)) base[hc * NT] = w;
        hc += (lo > cut) | (hi > cut);
    }
    SV_DEV void safe(float lo, float hi, uint32_t w) {
        if ((lo > cut) | (hi > cut)) {
            if (hc < kPer) base[hc * NT] = w;
            ++hc;
        }
    }
};

template <typename E>
struct Core;

// bf16: running maximum on packed pairs, exponentials on f32 pairs.
template <>
struct Core<bf16_t> {
    static constexpr int VE = 8;
    using Key = uint32_t;
    using Col = PairCollect;
    struct St {
        uint32_t pm;
        float2 s0, s1;
    };
    SV_DEV static St init() { return St{0xFF80FF80u, make_float2(0.f, 0.f), make_float2(0.f, 0.f)}; }
    SV_DEV static float vmax(const uint4& v) {
        const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
        return fmaxf(bf_lo(m), bf_hi(m));
    }
    template <bool COL, typename C>
    SV_DEV static void vec(St& st, const uint4& v, float2 c2v, float2 nr2, C& col) {
        st.pm = bmax2(st.pm, bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)));
        float2 a0 = make_float2(bf_lo(v.x), bf_hi(v.x)), a1 = make_float2(bf_lo(v.y), bf_hi(v.y));
        float2 a2 = make_float2(bf_lo(v.z), bf_hi(v.z)), a3 = make_float2(bf_lo(v.w), bf_hi(v.w));
        if (COL) {
            if (col.hc <= PairCollect::kPer - 4) {  // room for the whole vector
                col.put(a0.x, a0.y, v.x);
                col.put(a1.x, a1.y, v.y);
                col.put(a2.x, a2.y, v.z);
                col.put(a3.x, a3.y, v.w);
            } else {
                col.safe(a0.x, a0.y, v.x);
                col.safe(a1.x, a1.y, v.y);
                col.safe(a2.x, a2.y, v.z);
                col.safe(a3.x, a3.y, v.w);
            }
        }
        a0 = __ffma2_rn(a0, c2v, nr2);
        a1 = __ffma2_rn(a1, c2v, nr2);
        a2 = __ffma2_rn(a2, c2v, nr2);
        a3 = __ffma2_rn(a3, c2v, nr2);
        a0.x = ex2(a0.x);
        a0.y = ex2(a0.y);
        a1.x = ex2(a1.x);
        a1.y = ex2(a1.y);
        a2.x = ex2(a2.x);
        a2.y = ex2(a2.y);
        a3.x = ex2(a3.x);
        a3.y = ex2(a3.y);
        st.s0 = __fadd2_rn(st.s0, a0);
        st.s1 = __fadd2_rn(st.s1, a1);
        st.s0 = __fadd2_rn(st.s0, a2);
        st.s1 = __fadd2_rn(st.s1, a3);
    }
    template <bool COL, typename C>
    SV_DEV static void one(St& st, const bf16_t* p, float c2, float nref, C& col) {
        const uint32_t raw = __ldg(reinterpret_cast<const unsigned short*>(p));
        st.pm = bmax2(st.pm, raw | (raw << 16));
        const float x = __uint_as_float(raw << 16);
        if (COL) col.safe(x, -INFINITY, raw | 0xFF800000u);  // the other half -inf
        st.s0.x += ex2(fmaf(x, c2, nref));
    }
    SV_DEV static float maxof(const St& st) { return max_nan(bf_lo(st.pm), bf_hi(st.pm)); }
    SV_DEV static float sumof(const St& st) {
        const float2 t = __fadd2_rn(st.s0, st.s1);
        return t.x + t.y;
    }
};

// fp32: exponentials on pairs.
template <>
struct Core<float> {
    static constexpr int VE = 4;
    using Key = uint32_t;
    using Col = Collect<uint32_t>;
    struct St {
        float pm;
        float2 s0, s1;
    };
    SV_DEV static St init() { return St{-INFINITY, make_float2(0.f, 0.f), make_float2(0.f, 0.f)}; }
    SV_DEV static float vmax(const uint4& v) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    template <bool COL, typename C>
    SV_DEV static void vec(St& st, const uint4& v, float2 c2v, float2 nr2, C& col) {
        float2 a0 = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        float2 a1 = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
        st.pm = max_nan(st.pm, max_nan(max_nan(a0.x, a0.y), max_nan(a1.x, a1.y)));
        if (COL) {
            col(a0.x, v.x);
            col(a0.y, v.y);
            col(a1.x, v.z);
            col(a1.y, v.w);
        }
        a0 = __ffma2_rn(a0, c2v, nr2);
        a1 = __ffma2_rn(a1, c2v, nr2);
        a0.x = ex2(a0.x);
        a0.y = ex2(a0.y);
        a1.x = ex2(a1.x);
        a1.y = ex2(a1.y);
        st.s0 = __fadd2_rn(st.s0, a0);
        st.s1 = __fadd2_rn(st.s1, a1);
    }
    template <bool COL, typename C>
    SV_DEV static void one(St& st, const float* p, float c2, float nref, C& col) {
        const float x = __ldg(p);
        st.pm = max_nan(st.pm, x);
        if (COL) col(x, __float_as_uint(x));
        st.s0.x += ex2(fmaf(x, c2, nref));
    }
    SV_DEV static float maxof(const St& st) { return st.pm; }
    SV_DEV static float sumof(const St& st) {
        const float2 t = __fadd2_rn(st.s0, st.s1);
        return t.x + t.y;
    }
};

struct RowStats {
    float m;     // row (segment) maximum, NaN if any logit is NaN
    float sref;  // sum of exp2((z - ref) c2)
    float ref;
};

// Streams elements [i0, i1) of row: maximum and sum against a fixed
// reference (the first group's maximum when ref_in is NaN). Every thread of
// the CTA must call it; all return the same statistics. With COL, logits
// above ref - wc go to the thread's key slots.
template <typename E, bool COL>
__device__ __noinline__ RowStats stream_row(Shared& s, const E* row, int i0, int i1, float c2, float wc,
                                            float ref_in) {
    using C = Core<E>;
    constexpr int VE = C::VE;
    constexpr int es = sizeof(E);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uintptr_t addr = (uintptr_t)(row + i0);
    const int head = min(i1 - i0, (int)(((16 - (addr & 15)) & 15) / es));
    const int base = i0 + head;
    const int nb = (i1 - base) / VE;
    const uint4* vp = reinterpret_cast<const uint4*>(row + base);
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (tid + u * NT < nb) v[u] = ld_stream_v4(vp + tid + u * NT);
    float ref = ref_in;
    if (ref_in != ref_in) {
        float vm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (tid + u * NT < nb) vm = fmaxf(vm, C::vmax(v[u]));
        for (int o = 16; o; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, o));
        if (lane == 0 && vm > -INFINITY) atomicMax(&s.hmax, f32_key(vm));
        __syncthreads();
        ref = key_to_f32(s.hmax);
        if (!(ref > -INFINITY && ref < INFINITY)) ref = 0.f;
    }
    const float nref = -(ref * c2);
    const float2 c2v = make_float2(c2, c2), nr2 = make_float2(nref, nref);
    typename C::St st = C::init();
    using K = typename C::Key;
    typename C::Col col{reinterpret_cast<K*>(s.u.slots) + tid, ref - wc, 0};
    if (tid < head) C::template one<COL>(st, row + i0 + tid, c2, nref, col);
#pragma unroll
    for (int u = 0; u < kU; ++u)
        if (tid + u * NT < nb) C::template vec<COL>(st, v[u], c2v, nr2, col);
    for (int j = tid + NT * kU; j < nb; j += NT * kU) {
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (j + u * NT < nb) v[u] = ld_stream_v4(vp + j + u * NT);
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (j + u * NT < nb) C::template vec<COL>(st, v[u], c2v, nr2, col);
    }
    const int t = base + nb * VE + tid;
    if (t < i1) C::template one<COL>(st, row + t, c2, nref, col);
    if (COL) {
        s.hn[tid] = (unsigned short)min(col.hc, C::Col::kPer);
        if (col.hc > C::Col::kPer) s.ovf = 1;
        if (tid == 0) s.cut = ref - wc;
    }
    // block reduction: maximum (NaN-propagating), sum in a fixed order
    float tm = C::maxof(st), ts = C::sumof(st);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        tm = max_nan(tm, __shfl_xor_sync(0xFFFFFFFFu, tm, o));
        ts += __shfl_xor_sync(0xFFFFFFFFu, ts, o);
    }
    if (lane == 0) {
        s.red_m[warp] = tm;
        s.red_s[warp] = ts;
    }
    __syncthreads();
    RowStats r{s.red_m[0], s.red_s[0], ref};
    for (int w = 1; w < NW; ++w) {
        r.m = max_nan(r.m, s.red_m[w]);
        r.sref += s.red_s[w];
    }
    __syncthreads();
    return r;
}

// (m, S) of elements [i0, i1) with S against m: S = sref 2^((ref - m) c2),
// summed again against m when the sum against the reference left the fp32
// range. Every thread of the CTA must call it.
template <typename E, bool COL>
SV_DEV RowStats row_stats(Shared& s, const E* row, int i0, int i1, float c2, float wc) {
    RowStats r = stream_row<E, COL>(s, row, i0, i1, c2, wc, NAN);
    if (r.m > -INFINITY && r.m < INFINITY) {
        if (r.sref > 0.f && r.sref <= 3.0e38f) {
            r.sref *= ex2((r.ref - r.m) * c2);
        } else {
            const RowStats q = stream_row<E, false>(s, row, i0, i1, c2, wc, r.m);
            r.sref = q.sref;
        }
    }
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
        rr.has_x = r < p.gamma && p.draft_tokens != nullptr;  // records without tokens: no test
    } else {
        rr.k = r - p.gamma - 1;
        rr.ptr = reinterpret_cast<const E*>(p.draft) + ((size_t)b * p.gamma + rr.k) * p.V;
        rr.has_x = p.draft_tokens != nullptr;
    }
    return rr;
}


// Threshold of a bf16 row from its stored keys counted per distinct value
// (bin j holds the values of ordinal ord16(m) - j, largest first; the cut was
// fixed for the row, so the stored values form an upper set). Warp 0 scans
// the bins in use; the bins are cleared again before returning. False when
// the stored keys do not decide the threshold. Every thread must call it.
__device__ __noinline__ bool bf16_threshold(Shared& s, const RowParams& p, float m, float S, float* thr,
                                            float* sk) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float c2 = p.c2, mc = m * c2;
    const int top = (int)ord16(__float_as_uint(m) >> 16);  // every stored key is <= m
    if (s.odirty) {  // the binned selection has used this storage: clear every bin once
        for (int j = tid; j < kOrd; j += NT) s.h.ocnt[j] = 0u;
        __syncthreads();
        if (tid == 0) s.odirty = 0;
    }
    const uint32_t* slots = reinterpret_cast<const uint32_t*>(s.u.slots);
    const int n = s.hn[tid];
    const float cut = s.cut;
    int jm = -1;
    auto count = [&](uint32_t raw) {
        if (__uint_as_float(raw << 16) > cut) {
            const int j = top - (int)ord16(raw);
            if (j < kOrd) {
                atomicAdd(&s.h.ocnt[j], 1u);
                jm = max(jm, j);
            }  // below it: not needed, the counted values stay an upper set
        }
    };
    for (int c = 0; c < n; ++c) {
        const uint32_t w = slots[c * NT + tid];
        count(w & 0xFFFFu);
        count(w >> 16);
    }
    jm = __reduce_max_sync(0xFFFFFFFFu, jm);
    if (lane == 0 && jm >= 0) atomicMax(&s.jmax, jm);
    __syncthreads();
    const int jz = s.jmax;
    // every thread owns a few consecutive bins; an exclusive scan of (count,
    // mass) in thread order gives each thread its running weights
    const int nbins = jz + 1;
    const int per = (nbins + NT - 1) / NT;
    const int j0 = min(nbins, tid * per), j1 = min(nbins, j0 + per);
    auto mass_of = [&](int j, unsigned c) {
        return (unsigned long long)c * fx_of(fmaf(ord16_value((uint32_t)(top - j)), c2, -mc));
    };
    unsigned long long tc = 0ull, tw = 0ull;
    for (int j = j0; j < j1; ++j) {
        const unsigned c = s.h.ocnt[j];
        if (c) {
            tc += c;
            tw += mass_of(j, c);
        }
    }
    unsigned long long ic = tc, iw = tw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long yc = __shfl_up_sync(0xFFFFFFFFu, ic, d);
        const unsigned long long yw = __shfl_up_sync(0xFFFFFFFFu, iw, d);
        if (lane >= d) {
            ic += yc;
            iw += yw;
        }
    }
    if (lane == 31) {
        s.ured[warp] = ic;
        s.ured2[warp] = iw;
    }
    if (tid == 0) s.bi[5] = -1;
    __syncthreads();
    unsigned long long ec = ic - tc, ew = iw - tw;
    for (int w = 0; w < warp; ++w) {
        ec += s.ured[w];
        ew += s.ured2[w];
    }
    // the first non-empty bin j <= jlim whose running weight reaches target:
    // found by the one thread whose bins hold it
    auto find = [&](bool by_count, unsigned long long target, int jlim, int* jo, unsigned long long* wo) {
        if ((by_count ? ec : ew) < target) {
            unsigned long long c = ec, w = ew;
            for (int j = j0; j < j1 && j <= jlim; ++j) {
                const unsigned k = s.h.ocnt[j];
                if (!k) continue;
                c += k;
                w += mass_of(j, k);
                if ((by_count ? c : w) >= target) {
                    s.bi[5] = j;
                    s.ured[NW] = w;
                    break;
                }
            }
        }
        __syncthreads();
        *jo = s.bi[5];
        *wo = s.ured[NW];
        __syncthreads();
        if (tid == 0) s.bi[5] = -1;
        return *jo >= 0;
    };
    unsigned long long kept = (unsigned long long)(S * kFx);
    float t = -INFINITY;
    int jk = nbins - 1;
    bool ok = true;
    if (p.transform & kXfTopK) {
        unsigned long long w;
        ok = find(true, (unsigned long long)p.top_k, nbins - 1, &jk, &w);
        if (ok) {
            t = ord16_value((uint32_t)(top - jk));
            kept = w;
        }
    }
    if (ok && (p.transform & kXfTopP)) {
        int j;
        unsigned long long w;
        if (p.transform & kXfTopK) __syncthreads();  // s.bi[5] reset before the second search
        ok = find(false, top_p_target(p.top_p, kept), jk, &j, &w);
        if (ok) {
            t = ord16_value((uint32_t)(top - j));
            kept = w;
        }
    }
    *thr = t;
    *sk = (float)kept * (1.0f / kFx);
    for (int j = tid; j <= jz; j += NT) s.h.ocnt[j] = 0u;  // clean for the next row
    if (tid == 0) s.jmax = -1;
    return ok;
}

// bf16 rows: stores the candidate pairs of the row again, with a cut below
// its finished maximum (a second, wider collection when the keys stored
// while streaming do not decide the threshold or overflowed). Four 16-byte
// vectors in flight per thread; the 32-bit word of each adjacent pair with a
// logit above the cut goes to the thread's slots. Every thread must call it;
// it sets s.hn, s.cut and s.ovf.
SV_DEV void recollect_bf16(Shared& s, const bf16_t* row, int V, float cut) {
    const int tid = threadIdx.x;
    const unsigned short* rs = reinterpret_cast<const unsigned short*>(row);
    __syncthreads();  // every thread is past its last use of the slots and the flag
    if (tid == 0) {
        s.ovf = 0;
        s.cut = cut;
    }
    PairCollect col{reinterpret_cast<uint32_t*>(s.u.slots) + tid, cut, 0};
    const int head = min(V, (int)(((16 - ((uintptr_t)row & 15)) & 15) / 2));
    if (tid < head) {
        const uint32_t raw = __ldg(rs + tid);
        col.safe(__uint_as_float(raw << 16), -INFINITY, raw | 0xFF800000u);
    }
    const int nb = (V - head) / 8;
    const uint4* vp = reinterpret_cast<const uint4*>(row + head);
    for (int j = tid; j < nb; j += NT * kU) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (j + u * NT < nb) v[u] = __ldcg(vp + j + u * NT);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (j + u * NT < nb) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) col.safe(bf_lo(w[q]), bf_hi(w[q]), w[q]);
            }
        }
    }
    const int t = head + nb * 8 + tid;
    if (t < V) {
        const uint32_t raw = __ldg(rs + t);
        col.safe(__uint_as_float(raw << 16), -INFINITY, raw | 0xFF800000u);
    }
    __syncthreads();  // the flag's reset before any thread sets it
    s.hn[tid] = (unsigned short)min(col.hc, PairCollect::kPer);
    if (col.hc > PairCollect::kPer) s.ovf = 1;
    __syncthreads();
}

// Threshold and kept mass of a row: from the stored keys when they decide it,
// else from the row in global memory.
template <typename E>
__device__ __noinline__ void row_threshold(Shared& s, const RowParams& p, const E* row, float ref, float m,
                                           float S, bool use_slots, float* thr, float* sk) {
    const int tid = threadIdx.x;
    const float c2 = p.c2, mc = m * c2;
    constexpr int npass = sizeof(E) == 4 ? 4 : 2;
    if constexpr (sizeof(E) == 2) {
        if (use_slots) {
            // the stored pairs hold every value above the cut. Slots that
            // overflowed are filled again with the same window below the
            // finished maximum (tighter than below the reference); a window
            // that held too little is widened; then the selection over the
            // whole row
            if (!s.ovf && bf16_threshold(s, p, m, S, thr, sk)) return;
            if (s.ovf) {
                recollect_bf16(s, row, p.V, m - (float)(kWinB + 1) / c2);
                if (!s.ovf && bf16_threshold(s, p, m, S, thr, sk)) return;
            }
            recollect_bf16(s, row, p.V, m - (float)(kWinWide + 1) / c2);
            if (!s.ovf && bf16_threshold(s, p, m, S, thr, sk)) return;
        }
    } else if (use_slots && !s.ovf) {
        using K = typename Core<E>::Key;
        const K* slots = reinterpret_cast<const K*>(s.u.slots);
        const int n = s.hn[tid];
        const int nmax = __reduce_max_sync(0xFFFFFFFFu, n);
        auto each = [&](auto f) {
            for (int c = 0; c < nmax; ++c) {
                const bool v0 = c < n;
                const uint32_t raw = v0 ? (uint32_t)slots[c * NT + tid] : 0u;
                const float z = sizeof(E) == 2 ? __uint_as_float(raw << 16) : __uint_as_float(raw);
                const float a = v0 ? fmaf(z, c2, -mc) : -INFINITY;
                f(v0 && a > -(float)kWin, f32_key(z), a);
            }
        };
        if (threshold_from<true>(s, p, each, npass, true, S, thr, sk)) return;
    }
    const int V = p.V;
    auto each = [&](auto f) {
        for (int base = 0; base < V; base += NT) {
            const int i = base + tid;
            const bool v = i < V;
            const float z = v ? VecTraits<E>::load1(row + i) : -INFINITY;
            f(v, f32_key(z), fmaf(z, c2, -mc));
        }
    };
    threshold_from<false>(s, p, each, npass, false, S, thr, sk);
}

// --- per-row draw (sampling) and per-sequence resolve (verification) --------

// One draw per row from its transformed probabilities, straight after the
// row's statistics (the row is still in L2).
template <typename E>
__device__ __noinline__ void sample_row(Shared& s, const RowParams& p, const E* row, int b, int r, int rowid) {
    const RowRec rec = s.u.rec[0];
    int tok = -1;
    if (!(rec.flags & kRecEData)) {
        const float u = uniform01(p.seed, p.offset + (uint64_t)b, p.pos0 + (uint32_t)r, p.purpose);
        tok = draw_q<E>(s.draw, row, p.V, rec, p.c2, u);
    }
    if (threadIdx.x == 0) {
        if (SV_IN(rowid, (long long)p.B * p.rows_per_b)) p.sample_out[rowid] = tok;
        if (tok < 0 && p.status) atomicMax(&p.status[b], kEData);
    }
}

// Sequence b, once all its rows have records: acceptance left to right up to
// the first rejection n, then the outputs except the one drawn token (the
// residual of position n, or the bonus token from q_gamma), which the draw
// kernel below writes; n (or -1 for a sequence with bad data) is left in
// p.seq_n[b]. With lenience l the test is u < q/(l p) (the lenient variant
// of "Fast Inference from Transformers via Speculative Decoding", method
// details, extension of its appendix F); l = 1 is the exact method.
template <typename E>
__device__ __noinline__ void resolve_sequence(Shared& s, const RowParams& p, int b) {
    const int tid = threadIdx.x;
    const int R = p.rows_per_b, G = p.gamma;
    __threadfence();
    for (int i = tid; i < R; i += NT)
        if (SV_IN(i, kMaxRows)) s.u.rec[i] = load_rec(p.rows + (size_t)b * R + i);
    __syncthreads();
    if (tid == 0) {
        int flags = 0;
        for (int i = 0; i < R; ++i) flags |= s.u.rec[i].flags;
        int n = G;
        for (int k = 0; k < G; ++k) {
            const RowRec& t = s.u.rec[k];
            const RowRec& d = s.u.rec[G + 1 + k];
            const float q = KeptExp{t.thr, p.c2, t.m * p.c2, 1.f}(t.zx) / t.Sk;
            const float pd = KeptExp{d.thr, p.c2, d.m * p.c2, 1.f}(d.zx) / d.Sk;
            if (p.probs_dbg) {
                p.probs_dbg[((size_t)b * G + k) * 2 + 0] = q;
                p.probs_dbg[((size_t)b * G + k) * 2 + 1] = pd;
            }
            if (n == G) {
                const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
                if (!accept_test(u, q, p.lenience * pd)) n = k;
            }
        }
        const int stt = (flags & kRecEData) ? kEData : kOk;
        p.accepted[b] = stt ? -1 : n;
        p.seq_n[b] = stt ? -1 : n;
        if (stt) p.next_token[b] = -1;
        if (p.status) p.status[b] = stt;
        s.bi[2] = n;
        s.bi[3] = stt;
    }
    __syncthreads();
    const int n = s.bi[2], stt = s.bi[3];
    for (int j = tid; j <= G; j += NT)
        if ((stt || j != n) && SV_IN_SEQ((size_t)b * (G + 1) + j, (long long)p.B * (G + 1), p.status, b))
            p.tokens[(size_t)b * (G + 1) + j] = (!stt && j < n) ? s.u.rec[j].x : -1;
}

// One draw per resolved sequence: the residual max(0, q_n - l p_n) after a
// rejection at n, or the bonus token from q_gamma (with the same inverse CDF
// as every other draw). Persistent CTAs take sequences from a counter; many
// sequences are drawn at once, so the rounds' memory latency overlaps.
template <typename E>
__global__ void __launch_bounds__(NT, sizeof(E) == 4 ? 4 : 6) draw_kernel(const __grid_constant__ RowParams p) {
    __shared__ DrawShared ds;
    __shared__ RowRec rec[2];
    __shared__ int job;
    const int tid = threadIdx.x;
    const int R = p.rows_per_b, G = p.gamma;
    unsigned* counter = p.work + 1;
    for (;;) {
        if (tid == 0) job = (int)atomicAdd(counter, 1u);
        __syncthreads();
        const int b = job;
        if (b >= p.B) break;
        const int n = p.seq_n[b];
        if (n >= 0 && SV_IN_SEQ(n, G + 1, p.status, b)) {
            if (tid == 0) rec[0] = load_rec(p.rows + (size_t)b * R + n);
            if (tid == 1 && n < G) rec[1] = load_rec(p.rows + (size_t)b * R + G + 1 + n);
            __syncthreads();
            const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)n, kPurposeResample);
            const E* rt = row_ref<E>(p, b, n).ptr;
            int tok;
            if (n < G)
                tok = draw_residual<E, draw_vec<E>()>(ds, rt, row_ref<E>(p, b, G + 1 + n).ptr, p.V, rec[0], rec[1],
                                                 p.c2, u2, p.lenience);
            else
                tok = draw_q<E, draw_vec<E>()>(ds, rt, p.V, rec[0], p.c2, u2);
            if (tid == 0) {
                p.next_token[b] = tok;
                p.tokens[(size_t)b * (G + 1) + n] = tok;
            }
        }
        __syncthreads();
    }
}

// L2 prefetch of the 16-byte-aligned interior of elements [i0, i1) of row
// when it is at most kPrefetchBytes (a hint: no data moves into the SM).
// Longer units are not prefetched: across all CTAs they would exceed L2.
template <typename E>
SV_DEV void prefetch_l2(const E* row, int i0, int i1) {
    const uintptr_t a = ((uintptr_t)(row + i0) + 15) & ~(uintptr_t)15;
    const uintptr_t e = (uintptr_t)(row + i1) & ~(uintptr_t)15;
    if (e > a && e - a <= kPrefetchBytes)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"((uint32_t)(e - a)) : "memory");
}

// --- the kernel -----------------------------------------------------------------

template <typename E, bool XF>
__global__ void __launch_bounds__(NT, 5) row_kernel(const __grid_constant__ RowParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Shared& s = *reinterpret_cast<Shared*>(smem_raw);
    const int tid = threadIdx.x;
    const int R = p.rows_per_b;
    const int nunits = p.B * R * p.nseg;
    const bool col = XF && p.nseg == 1;
    const float wc = (float)((sizeof(E) == 2 ? kWinB : kWin) + 1) / p.c2;
    auto locate = [&](int u, int* b, int* r, int* i0, int* i1) {
        const int rowid = u / p.nseg, seg = u - rowid * p.nseg;
        *b = rowid / R;
        *r = rowid - *b * R;
        *i0 = seg * p.seg_len;
        *i1 = min(p.V, *i0 + p.seg_len);
    };
    if (tid == 0) {
        s.odirty = 1;
        s.jmax = -1;
        s.q[0] = (int)atomicAdd(p.work, 1u);
        s.q[1] = (int)atomicAdd(p.work, 1u);
        s.hmax = kKeyNegInf;
        s.ovf = 0;
    }
    for (int it = 0;; ++it) {
        __syncthreads();
        const int unit = s.q[it % 3];
        if (unit >= nunits) break;
        unsigned pre = 0u;
        if (tid == 0) {
            pre = atomicAdd(p.work, 1u);  // the unit after next, fetched while this one streams
            // a short next unit moves from HBM into L2 while this one streams
            const int nxt = s.q[(it + 1) % 3];
            if (nxt < nunits) {
                int b2, r2, j0, j1;
                locate(nxt, &b2, &r2, &j0, &j1);
                prefetch_l2(row_ref<E>(p, b2, r2).ptr, j0, j1);
            }
        }
        const int rowid = unit / p.nseg;
        int b, r, i0, i1;
        locate(unit, &b, &r, &i0, &i1);
        const RowRef<E> rr = row_ref<E>(p, b, r);
        // the draft token and its logit in this row (loaded early, used at the end)
        int x = -1;
        float zx = 0.f;
        if (tid == 0 && rr.has_x) {
            if (SV_IN((size_t)b * p.gamma + rr.k, (long long)p.B * p.gamma)) x = p.draft_tokens[(size_t)b * p.gamma + rr.k];
            if (x >= i0 && x < i1) zx = VecTraits<E>::load1(rr.ptr + x);
        }

        const RowStats st = col ? row_stats<E, true>(s, rr.ptr, i0, i1, p.c2, wc)
                                : row_stats<E, false>(s, rr.ptr, i0, i1, p.c2, wc);
        if (tid == 0) {
            s.q[(it + 2) % 3] = (int)pre;
            s.hmax = kKeyNegInf;
        }

        // ---- row record (by the last segment of the row to finish) ----
        bool have_row = p.nseg == 1;
        float m = st.m, S = st.sref;
        if (p.nseg > 1) {
            if (tid == 0) {
                SegRec sr;
                sr.m = m;
                sr.s = S;
                sr.zx = zx;
                sr.flags = 0;
                if (SV_IN(unit, nunits)) p.segs[unit] = sr;
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
            const bool bad = !(m > -INFINITY && m < INFINITY);
            float thr = -INFINITY, sk = S;
            if (XF && !bad) row_threshold<E>(s, p, rr.ptr, st.ref, m, S, col, &thr, &sk);
            __syncthreads();
            if (tid == 0) {
                RowRec rec;
                rec.m = m;
                rec.S = S;
                rec.thr = thr;
                rec.Sk = sk;
                rec.zx = zx;
                rec.x = x;
                rec.flags = (bad || (rr.has_x && (x < 0 || x >= p.V))) ? kRecEData : 0;
                rec.nkept = -1;
                if (SV_IN(rowid, (long long)p.B * R)) p.rows[rowid] = rec;
                s.u.rec[0] = rec;
                s.ovf = 0;
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

template <typename E>
cudaError_t launch_draws_t(const RowParams& p, int sms, cudaStream_t stream) {
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draw_kernel<E>, NT, 0) != cudaSuccess || n < 1) n = 1;
        return n;
    }();
    const int grid = (int)std::min<long long>(p.B, (long long)sms * per_sm);
    draw_kernel<E><<<grid, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rows(const RowParams& p, int dtype, int sms, cudaStream_t stream) {
    const bool xf = p.transform != 0;
    if (dtype == 0) return xf ? launch_t<float, true>(p, sms, stream) : launch_t<float, false>(p, sms, stream);
    return xf ? launch_t<bf16_t, true>(p, sms, stream) : launch_t<bf16_t, false>(p, sms, stream);
}

cudaError_t launch_draws(const RowParams& p, int dtype, int sms, cudaStream_t stream) {
    return dtype == 0 ? launch_draws_t<float>(p, sms, stream) : launch_draws_t<bf16_t>(p, sms, stream);
}

SV_DEBUG_READER(rows)

}  // namespace sv
