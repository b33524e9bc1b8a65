// Shared-memory row path: verification with a top-k / top-p transform on
// bf16 logits.
//
// The transforms of "Accelerating Large Language Model Decoding with
// Speculative Sampling" ("与标准采样方法的兼容性") need, for every row, an exact
// threshold tau (kept set {z >= tau}) and the kept mass, on top of the
// maximum m and S = sum_i 2^((z_i - m) log2e / T). One persistent CTA per SM
// keeps a ring of nbuf row buffers in shared memory and gives each step of a
// row to its own warps, which meet only at mbarriers, so that warps of
// different rows run at once and no step waits for a CTA-wide barrier:
//
//   copy lane     stages whole rows into the ring with bulk asynchronous
//                 copies (the TMA engine, non-tensor form), a buffer as soon
//                 as it is released, and prefetches later rows into L2;
//   max warps     (kMaxWarps) the row maximum (packed bf16x2 maxima, one
//                 shared atomic per warp), a row ahead of the sum warps;
//   sum warps     two groups of kGroupWarps taking alternate rows (while
//                 one group sums, the other gathers or waits); in its group
//                 each warp owns a contiguous range of the row: S against m,
//                 the vectors holding a logit within kWin octaves of m listed
//                 in index order, then those logits gathered, counted per
//                 distinct bf16 value below m and, for a target row, written
//                 as the warp's region of the row's window list;
//   select warps  one per ring slot: from the counts, the exact top-k /
//                 top-p threshold and kept mass; the row record.
//
// A row whose window does not decide the threshold (a list overflowed, or
// the crossing lies deeper than kWin octaves) is queued and its record
// marked; smem_tail_kernel then counts such a row per distinct bf16 value
// over a thread-block cluster (the same threshold as select.cuh's selection)
// while its other warps do the per-sequence work: acceptance at every
// position ("改进的拒绝采样"), the first rejection n, and the one draw from
// max(0, q_n - l p_n) or the bonus draw from q_gamma, one warp per sequence
// over the window list of target row n. A sequence with a marked row, or
// without a usable list, is resolved last from the rows by
// smem_fulldraw_kernel.

#include <cooperative_groups.h>

#include "common.cuh"
#include "draw.cuh"
#include "select.cuh"

namespace sv {
namespace {

using namespace sel;

constexpr int NT = kSelNT;               // tail and full-row draw kernels
constexpr int NW = NT / 32;
constexpr int kWin = 12;                 // candidates: logits within kWin octaves of the row maximum
constexpr int kGroupWarps = kKeptRegions;  // sum warps per group (one window-list region each)
constexpr int kSumWarps = 2 * kGroupWarps;
constexpr int kMaxWarps = 4;
constexpr int kMaxSlots = 3;             // deepest ring (one select warp per slot)
constexpr int kMaxWarp0 = kSumWarps;     // warp index of the first max warp
constexpr int kSelWarp0 = kMaxWarp0 + kMaxWarps;
constexpr int kCopyWarp = kSelWarp0 + kMaxSlots;
constexpr int kRowThreads = 32 * (kCopyWarp + 1);
constexpr int kListCap = 128;            // vectors listed per sum warp and row
constexpr int kElemCap = kKeptRegionCap; // window logits gathered per sum warp and row
constexpr int kOrdBins = 1024;           // distinct bf16 values below the maximum counted
constexpr int kPrefetchAhead = 2;        // rows prefetched into L2 ahead of their copies
constexpr uint32_t kChunk = 32768;       // bytes per bulk copy or prefetch
#ifdef SPEC_DEBUG
static __device__ int g_withhold = -1;   // spec_debug_withhold_copy
#endif
constexpr uint32_t kSuspendNs = 20000;   // longest suspension of one poll of a wait
constexpr uint32_t kWaitPolls = 1u << 16;  // polls before a wait gives up (about a second)
constexpr unsigned kKeyNaN = 0xFFFFu;    // row maximum key of a row holding a NaN

// ---- mbarrier, bulk copies ------------------------------------------------------

SV_DEV uint32_t smem_u32(const void* ptr) { return (uint32_t)__cvta_generic_to_shared(ptr); }

SV_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

SV_DEV void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

SV_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

SV_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

SV_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete is suspended
// (it takes no issue slots) until the phase completes or kSuspendNs pass.
SV_DEV bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier to complete; false after
// kWaitPolls suspended polls or once `abort` is set.
SV_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort) {
    for (uint32_t it = 0; it < kWaitPolls; ++it) {
        if (mbar_try_wait_suspend(bar, parity)) return true;
        if (abort && *abort) return false;
    }
    return false;
}

// Global -> L2 only (a hint: nothing moves into the SM).
SV_DEV void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Orders the CTA's earlier shared-memory accesses before bulk copies issued next.
SV_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Global -> this CTA's shared memory; both addresses 16-byte aligned, bytes a
// multiple of 16; completion is counted on `bar`.
SV_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- shared state -----------------------------------------------------------------

// One row in flight. The max warps fold the row maximum into mkey (the
// bf16 ordinal of m, kKeyNaN for a NaN) and leave the draft token; each sum
// warp leaves its sum and adds the row's window logits to the counts per
// ordinal below m. The sum warps' part comes in two sets that alternate
// with the slot's uses, so that the select warp may still read one while
// the next use fills the other; the select warp clears what it used.
struct SlotSet {
    float reds[kGroupWarps];                 // per-warp sums (warps of the row's group)
    int wjm[kGroupWarps];                    // per-warp deepest ordinal offset (-1: none)
    int cn[kGroupWarps];                     // per-warp window logits (kElemCap + 1: more than its region
                                             // holds; -1: its vector list overflowed, counts incomplete)
    uint32_t bins[kOrdBins / 2];             // window logits per ordinal below m, two 16-bit counts a word
};
struct Slot {
    unsigned mkey;
    int x;                                   // the draft token (-1: none)
    float zx;                                // its logit
    SlotSet set[2];
};
constexpr size_t kSlotBytes = (sizeof(Slot) + 127) & ~(size_t)127;
constexpr size_t kListBytes = (size_t)kSumWarps * kListCap * sizeof(unsigned short);

// Row r of sequence b: target rows 0 .. gamma, then the gamma draft rows.
SV_DEV const unsigned short* row_src(const RowParams& p, int b, int r) {
    const int G = p.gamma;
    return r <= G ? reinterpret_cast<const unsigned short*>(p.target) + ((size_t)b * (G + 1) + r) * p.V
                  : reinterpret_cast<const unsigned short*>(p.draft) + ((size_t)b * G + (r - G - 1)) * p.V;
}

// The largest bf16 value not above x (x finite), duplicated in both halves.
SV_DEV uint32_t bf16_pair_down(float x) {
    const uint32_t b = __float_as_uint(x);
    uint32_t t = b & 0xFFFF0000u;
    if ((b & 0x80000000u) && (b & 0xFFFFu)) t += 0x10000u;  // negative: away from zero
    return t | (t >> 16);
}

SV_DEV float bf_raw(uint32_t raw) { return __uint_as_float(raw << 16); }

// The window of a row with maximum m: the logits above this bf16 pair (the
// largest bf16 at or below m - kWin octaves). It is closed upward, so it
// holds every logit at or above any logit in it.
SV_DEV uint32_t window_cut(float m, float width) { return bf16_pair_down(m - width); }

// Walks a CTA's rows j = j0, j0 + dj, ...: row = block + j grid, its
// sequence b and position r (row = b R + r), its ring slot s = j mod nbuf and
// the slot's use u = j div nbuf, advanced without divisions.
struct RowWalk {
    int row, b, r, s;
    uint32_t u;
    int drow, db, dr, ds, du, R, nbuf;
    SV_DEV RowWalk(int j0, int dj, int R_, int nbuf_) : R(R_), nbuf(nbuf_) {
        row = (int)blockIdx.x + j0 * (int)gridDim.x;
        b = row / R;
        r = row - b * R;
        s = j0 % nbuf;
        u = (uint32_t)(j0 / nbuf);
        drow = dj * (int)gridDim.x;
        db = drow / R;
        dr = drow - db * R;
        ds = dj % nbuf;
        du = dj / nbuf;
    }
    SV_DEV void next() {
        row += drow;
        b += db;
        r += dr;
        if (r >= R) {
            r -= R;
            ++b;
        }
        s += ds;
        u += (uint32_t)du;
        if (s >= nbuf) {
            s -= nbuf;
            ++u;
        }
    }
};

// The row maximum from its key.
SV_DEV float key_max(unsigned key) { return key == kKeyNaN ? __uint_as_float(0x7FC00000u) : ord16_value(key); }

// ---- selection by one warp -------------------------------------------------------

// The exact threshold from the window's logits counted per distinct bf16
// value: bin j holds the logits of ordinal ord16(m) - j, so bins run from
// the largest value down, and the mass of a bin is its count times the
// fixed-point mass of its value (the integers select.cuh sums element by
// element, so the two agree). Lane l owns the bins [l per, (l + 1) per): it
// totals them, a warp scan places the lanes, and the lane whose bins hold the
// crossing walks them. Top-k (by count) then top-p (by mass, over the kept
// bins). False when the window holds too few logits or too little mass to
// decide; else *thr, *sk (kept mass) and *jt (the crossing bin).
SV_DEV bool warp_threshold(const uint32_t* bins, int nb, int top, const RowParams& p, float mc, float S,
                           float* thr, float* sk, int* jt) {
    const int lane = threadIdx.x & 31;
    const float c2 = p.c2;
    const int per = (nb + 31) / 32;
    const int j0 = min(nb, lane * per), j1 = min(nb, j0 + per);
    const auto count_of = [&](int j) { return (bins[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu; };
    const auto mass_of = [&](int j, unsigned c) {
        return (unsigned long long)c * fx_of(fmaf(ord16_value((uint32_t)(top - j)), c2, -mc));
    };
    unsigned long long tc = 0ull, tw = 0ull;
    for (int j = j0; j < j1; ++j) {
        const unsigned c = count_of(j);
        if (c) {
            tc += c;
            tw += mass_of(j, c);
        }
    }
    unsigned long long ec = tc, ew = tw;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long yc = __shfl_up_sync(0xFFFFFFFFu, ec, d);
        const unsigned long long yw = __shfl_up_sync(0xFFFFFFFFu, ew, d);
        if (lane >= d) {
            ec += yc;
            ew += yw;
        }
    }
    ec -= tc;
    ew -= tw;
    // the first bin j <= jlim whose running weight reaches the target, and
    // the mass through it; -1 if none
    const auto find = [&](bool by_count, unsigned long long target, int jlim, unsigned long long* wo) {
        int hit = -1;
        unsigned long long hw = 0ull;
        if ((by_count ? ec : ew) < target) {
            unsigned long long c = ec, w = ew;
            for (int j = j0; j < j1 && j <= jlim; ++j) {
                const unsigned k = count_of(j);
                if (!k) continue;
                c += k;
                w += mass_of(j, k);
                if ((by_count ? c : w) >= target) {
                    hit = j;
                    hw = w;
                    break;
                }
            }
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, hit >= 0);
        if (!bal) return -1;
        const int src = __ffs(bal) - 1;
        *wo = __shfl_sync(0xFFFFFFFFu, hw, src);
        return __shfl_sync(0xFFFFFFFFu, hit, src);
    };
    unsigned long long kept = (unsigned long long)(S * kFx);
    int jk = nb - 1, j = -1;
    if (p.transform & kXfTopK) {
        unsigned long long w;
        jk = find(true, (unsigned long long)p.top_k, nb - 1, &w);
        if (jk < 0) return false;
        kept = w;
        j = jk;
    }
    if (p.transform & kXfTopP) {
        unsigned long long w;
        j = find(false, top_p_target(p.top_p, kept), jk, &w);
        if (j < 0) return false;
        kept = w;
    }
    *thr = ord16_value((uint32_t)(top - j));
    *sk = (float)kept * (1.0f / kFx);
    *jt = j;
    return true;
}

// ---- the row kernel -------------------------------------------------------------

// Rows are assigned to CTAs round-robin (row = block + j * grid); the CTA's
// j-th row goes through ring slot j mod nbuf. Per slot five mbarriers order
// the roles: full (the copy landed), maxed (the max warps are done), ready
// (the sum warps are done: sums, counts and gathered logits complete),
// empty (the buffer may be refilled), freed (the select warp is done with
// the slot). Every wait is bounded; a wait that gives up sets `abort`, after
// which every role stops, the rows not finished are recorded as timed out
// and the copies in flight are waited for.
__global__ void __launch_bounds__(kRowThreads, 1) smem_row_kernel(const __grid_constant__ RowParams p, const int nbuf) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ alignas(8) uint64_t full[kMaxSlots], maxed[kMaxSlots], ready[kMaxSlots], empty[kMaxSlots],
        hfree[kMaxSlots], freed[kMaxSlots][2];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = p.V, R = p.rows_per_b, G = p.gamma;
    const int nvec = V >> 3;
    const int nrows = p.B * R;  // below 2^30 (checked by the host)
    const float c2 = p.c2;
    const float width = (float)kWin / c2;  // the window in logit units
    const uint32_t bytes = (uint32_t)V * 2u;
    const size_t rb = ((size_t)bytes + 127) & ~(size_t)127;
    const unsigned lt = (1u << lane) - 1u;
    const auto slot_at = [&](int s) -> Slot& { return *reinterpret_cast<Slot*>(dyn + nbuf * rb + s * kSlotBytes); };
    volatile int* abort_v = &abort_flag;

    for (int s = 0; s < nbuf; ++s) {
        Slot& st = slot_at(s);
        for (int i = tid; i < kOrdBins; i += kRowThreads) st.set[i & 1].bins[i >> 1] = 0u;
        if (tid == 0) st.mkey = 0u;
    }
    if (tid == 0) {
        for (int s = 0; s < nbuf; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&maxed[s], kMaxWarps);
            mbar_init(&ready[s], kGroupWarps);
            mbar_init(&empty[s], kGroupWarps);
            mbar_init(&hfree[s], 1);
            mbar_init(&freed[s][0], 1);
            mbar_init(&freed[s][1], 1);
        }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp < kMaxWarp0) {
        // ---- sum warps: group g takes the rows j = g (mod 2); in it, warp
        // gw owns the vectors [v0, v1), balanced ----
        const int g = warp / kGroupWarps, gw = warp - g * kGroupWarps;
        const int v0 = (int)((long long)nvec * gw / kGroupWarps);
        const int v1 = (int)((long long)nvec * (gw + 1) / kGroupWarps);
        unsigned short* const list =
            reinterpret_cast<unsigned short*>(dyn + nbuf * (rb + kSlotBytes)) + warp * kListCap;
        for (RowWalk w(g, 2, R, nbuf);; w.next()) {
            const int row = w.row, s = w.s;
            if (row >= nrows) break;
            const uint32_t u = w.u;
            Slot& st = slot_at(s);
            const uint4* vr = reinterpret_cast<const uint4*>(dyn + s * rb);
            // the max warps saw the copy land and the slot freed
            bool ok = mbar_wait(&maxed[s], u & 1u, abort_v) && mbar_try_wait(&full[s], u & 1u);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) *abort_v = 1;
                break;
            }
            const float m = key_max(st.mkey);
            const bool bad = !(m > -INFINITY && m < INFINITY);

            // S against m, and the vectors holding a window logit listed in
            // ascending order (rounds of 32 consecutive vectors, lanes in
            // order)
            float S = 0.f;
            int nv = 0, cn = 0, jm = -1;
            if (!bad) {
                const float mc = m * c2;
                const float2 c2v = make_float2(c2, c2), nm = make_float2(-mc, -mc);
                const uint32_t cut2 = window_cut(m, width);
                float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
                const auto sum8 = [&](const uint4& xv) {
                    float2 a0 = __ffma2_rn(make_float2(bf_lo(xv.x), bf_hi(xv.x)), c2v, nm);
                    float2 a1 = __ffma2_rn(make_float2(bf_lo(xv.y), bf_hi(xv.y)), c2v, nm);
                    float2 a2 = __ffma2_rn(make_float2(bf_lo(xv.z), bf_hi(xv.z)), c2v, nm);
                    float2 a3 = __ffma2_rn(make_float2(bf_lo(xv.w), bf_hi(xv.w)), c2v, nm);
                    a0.x = ex2(a0.x);
                    a0.y = ex2(a0.y);
                    a1.x = ex2(a1.x);
                    a1.y = ex2(a1.y);
                    a2.x = ex2(a2.x);
                    a2.y = ex2(a2.y);
                    a3.x = ex2(a3.x);
                    a3.y = ex2(a3.y);
                    s0 = __fadd2_rn(s0, a0);
                    s1 = __fadd2_rn(s1, a1);
                    s0 = __fadd2_rn(s0, a2);
                    s1 = __fadd2_rn(s1, a3);
                };
                const auto note = [&](bool hit, int v) {
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, hit);
                    if (bal) {
                        const int at = nv + __popc(bal & lt);
                        if (hit && at < kListCap) list[at] = (unsigned short)v;
                        nv += __popc(bal);
                    }
                };
                const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
                int base = v0;
                for (; base + 32 <= v1; base += 32) {
                    const int va = base + lane;
                    const uint4 xa = vr[va];
                    const uint32_t ma = bmax2(bmax2(xa.x, xa.y), bmax2(xa.z, xa.w));
                    note(bmax2(ma, cut2) != cut2, va);
                    sum8(xa);
                }
                if (base < v1) {  // the last, partial round: missing vectors read as -inf
                    const int va = base + lane;
                    const uint4 xa = va < v1 ? vr[va] : ninf;
                    const uint32_t ma = bmax2(bmax2(xa.x, xa.y), bmax2(xa.z, xa.w));
                    note(bmax2(ma, cut2) != cut2, va);
                    sum8(xa);
                }
                const float2 t2 = __fadd2_rn(s0, s1);
                S = t2.x + t2.y;
#pragma unroll
                for (int o = 16; o; o >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);

                // the window logits of the listed vectors, counted per ordinal
                // below m and, for a target row, written as this warp's region
                // of the row's window list (index order: list order, lanes in
                // order, each lane's elements in order), once the select warp
                // is done with this set's previous use
                ok = u < 2 || mbar_wait(&freed[s][u & 1u], ((u >> 1) - 1u) & 1u, abort_v);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    if (lane == 0) *abort_v = 1;
                    break;
                }
                if (nv <= kListCap) {
                    const float cutf = bf_lo(cut2);
                    const int top = (int)ord16(__float_as_uint(m) >> 16);
                    const int b = w.b, r = w.r;
                    const bool tgt = r <= G && p.kept != nullptr;
                    const size_t rg = ((size_t)b * (G + 1) + (tgt ? r : 0)) * (size_t)p.kept_cap + gw * kElemCap;
                    uint32_t* const bins = st.set[u & 1u].bins;
                    for (int c0 = 0; c0 < nv; c0 += 32) {
                        const int i = c0 + lane;
                        unsigned em = 0u;
                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                        int v = 0;
                        if (i < nv) {
                            v = list[i];
                            if (SV_IN(v, nvec)) xv = vr[v];
                            em = (bf_lo(xv.x) > cutf) | (bf_hi(xv.x) > cutf) << 1 | (bf_lo(xv.y) > cutf) << 2 |
                                 (bf_hi(xv.y) > cutf) << 3 | (bf_lo(xv.z) > cutf) << 4 | (bf_hi(xv.z) > cutf) << 5 |
                                 (bf_lo(xv.w) > cutf) << 6 | (bf_hi(xv.w) > cutf) << 7;
                        }
                        // this lane's offset: the counts of the lanes below it, bit by bit
                        const unsigned cnt = __popc(em);
                        int o = cn;
#pragma unroll
                        for (int bit = 0; bit < 4; ++bit) {
                            const unsigned bb = __ballot_sync(0xFFFFFFFFu, (cnt >> bit) & 1u);
                            o += __popc(bb & lt) << bit;
                            cn += __popc(bb) << bit;
                        }
                        for (unsigned msk = em; msk; msk &= msk - 1u, ++o) {
                            const int e = __ffs(msk) - 1;
                            const uint32_t wd = e < 4 ? (e < 2 ? xv.x : xv.y) : (e < 6 ? xv.z : xv.w);
                            const uint32_t raw = e & 1 ? wd >> 16 : wd & 0xFFFFu;
                            const int jb = top - (int)ord16(raw);
                            jm = max(jm, jb);
                            if (jb < kOrdBins) atomicAdd(&bins[jb >> 1], 1u << ((jb & 1) * 16));
                            if (tgt && o < kElemCap && SV_IN(rg + o, (long long)p.B * (G + 1) * p.kept_cap)) {
                                p.kept[rg + o] = (uint32_t)(v * 8 + e) << 16 | raw;
                            }
                        }
                    }
                    jm = __reduce_max_sync(0xFFFFFFFFu, jm);
                    // more window logits than the region holds: the counts are
                    // complete, the row's window list is not
                    if (cn > kElemCap) cn = kElemCap + 1;
                    if (tgt && lane == 0 && SV_IN(rg / kElemCap, (long long)p.B * (G + 1) * kKeptRegions))
                        p.kept_cnt[rg / kElemCap] = (uint8_t)min(cn, 255);
                } else {
                    cn = -1;  // more listed vectors than the list holds: the counts are not complete
                }
            } else if (u >= 2 &&
                       !__all_sync(0xFFFFFFFFu, mbar_wait(&freed[s][u & 1u], ((u >> 1) - 1u) & 1u, abort_v))) {
                if (lane == 0) *abort_v = 1;
                break;
            }
            if (lane == 0) {
                SlotSet& ss = st.set[u & 1u];
                ss.reds[gw] = S;
                ss.cn[gw] = cn;
                ss.wjm[gw] = jm;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                mbar_arrive(&ready[s]);
            }
        }
    } else if (warp < kSelWarp0) {
        // ---- max warps: the row maximum, a quarter of the row each ----
        const int mw = warp - kMaxWarp0;
        const int v0 = (int)((long long)nvec * mw / kMaxWarps);
        const int v1 = (int)((long long)nvec * (mw + 1) / kMaxWarps);
        for (RowWalk w(0, 1, R, nbuf);; w.next()) {
            const int row = w.row, s = w.s;
            if (row >= nrows) break;
            const uint32_t u = w.u;
            Slot& st = slot_at(s);
            const uint4* vr = reinterpret_cast<const uint4*>(dyn + s * rb);
            const int b = w.b, r = w.r;
            const bool target = r <= G;
            const int k = target ? r : r - G - 1;
            const bool has_x = (!target || r < G) && p.draft_tokens != nullptr;
            // the draft token, loaded first (its latency overlaps the waits)
            int x = -1;
            if (mw == 0 && lane == 0 && has_x && SV_IN((size_t)b * G + k, (long long)p.B * G))
                x = __ldg(p.draft_tokens + (size_t)b * G + k);
            bool ok = mbar_wait(&full[s], u & 1u, abort_v);
            if (ok && u > 0) ok = mbar_wait(&hfree[s], (u - 1u) & 1u, abort_v);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) *abort_v = 1;
                break;
            }
            uint32_t pm = 0xFF80FF80u;
#pragma unroll 8
            for (int v = v0 + lane; v < v1; v += 32) {
                const uint4 xv = vr[v];
                pm = bmax2(pm, bmax2(bmax2(xv.x, xv.y), bmax2(xv.z, xv.w)));
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) pm = bmax2(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, o));
            if (lane == 0) {
                const float mv = max_nan(bf_lo(pm), bf_hi(pm));
                atomicMax(&st.mkey, mv != mv ? kKeyNaN : ord16(__float_as_uint(mv) >> 16));
                if (mw == 0) {
                    st.x = x;
                    st.zx = (has_x && x >= 0 && x < V) ? bf_raw(reinterpret_cast<const unsigned short*>(vr)[x]) : 0.f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&maxed[s]);
        }
    } else if (warp < kSelWarp0 + nbuf) {
        // ---- select warp of slot s ----
        const int s = warp - kSelWarp0;
        Slot& st = slot_at(s);
        for (RowWalk w(s, nbuf, R, nbuf);; w.next()) {
            const int row = w.row;
            if (row >= nrows) break;
            const uint32_t u = w.u;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ready[s], u & 1u, abort_v))) {
                // this slot's rows from here on are reported, unprocessed
                if (lane == 0) {
                    *abort_v = 1;
                    for (int rr = row; rr < nrows; rr += nbuf * (int)gridDim.x) {
                        RowRec rec = {};
                        rec.flags = kRecTimeout;
                        rec.x = -1;
                        rec.nkept = -1;
                        if (SV_IN(rr, nrows)) p.rows[rr] = rec;
                    }
                }
                break;
            }
            const int r = w.r;
            const bool target = r <= G;
            const bool has_x = (!target || r < G) && p.draft_tokens != nullptr;
            const float m = key_max(st.mkey);
            const bool bad = !(m > -INFINITY && m < INFINITY);
            const int x = st.x;
            const float zx = st.zx;
            __syncwarp();
            if (lane == 0) {
                // the max warps' part of the slot is free for its next row
                st.mkey = 0u;
                mbar_arrive(&hfree[s]);
            }
            // per-warp figures, lane w holding those of the row's group's warp w
            SlotSet& ss = st.set[u & 1u];
            const bool mine = lane < kGroupWarps;
            float S = mine ? ss.reds[lane] : 0.f;
            const int wcn = mine ? ss.cn[lane] : 0;
            int jm = mine ? ss.wjm[lane] : -1;
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
                jm = max(jm, __shfl_xor_sync(0xFFFFFFFFu, jm, o));
            }
            const bool fit = !bad && !__any_sync(0xFFFFFFFFu, wcn < 0) && jm >= 0 && jm < kOrdBins;
            float thr = -INFINITY, sk = S;
            int nkept = -1;
            bool decided = bad;
            const int top = (int)ord16(__float_as_uint(m) >> 16);
            int jt = 0;
            if (fit && warp_threshold(ss.bins, jm + 1, top, p, m * c2, S, &thr, &sk, &jt)) {
                decided = true;
                // a target row's window list (written by the sum warps) holds its kept set
                if (target && p.kept != nullptr && !__any_sync(0xFFFFFFFFu, wcn > kElemCap))
                    nkept = __reduce_add_sync(0xFFFFFFFFu, (unsigned)wcn);
            }
            if (lane == 0) {
                RowRec rec;
                rec.m = m;
                rec.S = S;
                rec.thr = thr;
                rec.Sk = sk;
                rec.zx = zx;
                rec.x = x;
                rec.flags = ((bad || (has_x && (x < 0 || x >= V))) ? kRecEData : 0) | (decided ? 0 : kRecFallback);
                rec.nkept = nkept;
                if (SV_IN(row, nrows)) p.rows[row] = rec;
                if (!decided) {
                    // the whole row decides it (fallback_rows, in smem_tail_kernel)
                    const unsigned qi = atomicAdd(p.work + 3, 1u);
                    if (SV_IN(qi, nrows)) p.fb_rows[qi] = row;
                }
            }
            // the counts cleared for the set's next use
            const int nw = (min(jm + 1, kOrdBins) + 1) >> 1;
            for (int i = lane; i < nw; i += 32) ss.bins[i] = 0u;
            __syncwarp();
            if (lane == 0) mbar_arrive(&freed[s][u & 1u]);
        }
    } else if (warp == kCopyWarp && lane == 0) {
        // ---- copy lane ----
        uint32_t issued = 0u;  // per slot s, bits 2s and 2s + 1: a copy issued, the parity of the last
        int jc = 0;
        for (RowWalk w(0, 1, R, nbuf); w.row < nrows; w.next(), ++jc) {
            const int s = w.s;
            const uint32_t u = w.u;
            if (u > 0 && !mbar_wait(&empty[s], (u - 1u) & 1u, abort_v)) {
                *abort_v = 1;
                break;
            }
#ifdef SPEC_DEBUG
            if (blockIdx.x == 0 && jc == g_withhold) continue;  // the buffer is never filled
#endif
            fence_proxy_async();
            mbar_expect_tx(&full[s], bytes);
            const char* src = reinterpret_cast<const char*>(row_src(p, w.b, w.r));
            unsigned char* dst = dyn + s * rb;
            for (uint32_t o = 0; o < bytes; o += kChunk) bulk_g2s(dst + o, src + o, min(kChunk, bytes - o), &full[s]);
            issued = (issued & ~(3u << (2 * s))) | ((1u | (u & 1u) << 1) << (2 * s));
            // a later row into L2, kPrefetchAhead copies ahead of its own copy
            // (the first copy prefetches the rows between)
            RowWalk q = w;
            const bool first = u == 0 && s == 0;
            for (int a = 0; a < (first ? nbuf : nbuf + kPrefetchAhead - 1); ++a) q.next();
            for (int a = 0; a < (first ? kPrefetchAhead : 1) && q.row < nrows; ++a, q.next()) {
                const char* ps = reinterpret_cast<const char*>(row_src(p, q.b, q.r));
                for (uint32_t o = 0; o < bytes; o += kChunk) prefetch_l2(ps + o, min(kChunk, bytes - o));
            }
        }
        // every copy issued lands before the CTA exits
        for (int s = 0; s < nbuf; ++s) {
            const uint32_t f = (issued >> (2 * s)) & 3u;
            if (f & 1u) mbar_wait(&full[s], f >> 1, nullptr);
        }
    }
    __syncwarp();  // the copy warp's lanes meet again before the CTA barrier
    __syncthreads();
}

// The queued rows: one thread-block cluster of kFbCluster CTAs per row
// (taken from a counter). The row's logits are counted per distinct bf16
// value (a 16-bit counter per value), the value range split over the
// cluster: CTA r reads the whole row (from L2 after the first reader) and
// counts the values of descending rank [r kFbRange, (r + 1) kFbRange). A
// value's mass is its count times the fixed-point mass of the value (the
// integers select.cuh sums element by element), so the threshold is the one
// of select.cuh's selection over the row. Each CTA totals its range (thread
// t owns kFbPer consecutive values, a block scan places the threads); the
// CTAs read one another's totals from distributed shared memory to place
// their ranges; the thread holding the crossing walks its values, and its
// CTA posts the result, which every CTA reads back through distributed
// shared memory. Completes the row's record (threshold and kept mass; no
// window list, so a draw from it reads the rows). Rows here are shorter than
// 65536, so no count reaches 2^16. All CTAs of a cluster take the same jobs
// and the same branches, so every cluster barrier completes.
constexpr int kFbValues = 65536;
constexpr int kFbCluster = 8;
constexpr int kFbRange = kFbValues / kFbCluster;  // values per CTA
constexpr int kFbPer = kFbRange / NT;             // values per thread
static_assert(kFbPer == 32, "one value per lane of a warp in the totals loop");

struct FallbackShared {
    unsigned long long wc[NW], ww[NW];  // block scan: per-warp totals
    unsigned long long cc, cw;          // this CTA's range totals (read by the cluster)
    int hit;                            // the crossing found in this CTA (descending rank), -1: none
    unsigned long long hw;              // the mass through it
    int job;                            // (rank 0) the row taken
};

// Inclusive scan of two 64-bit values in thread order over the CTA.
SV_DEV void block_scan2(FallbackShared& s, unsigned long long& a, unsigned long long& b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long ya = __shfl_up_sync(0xFFFFFFFFu, a, o);
        const unsigned long long yb = __shfl_up_sync(0xFFFFFFFFu, b, o);
        if (lane >= o) {
            a += ya;
            b += yb;
        }
    }
    __syncthreads();  // the previous scan's totals are read
    if (lane == 31) {
        s.wc[warp] = a;
        s.ww[warp] = b;
    }
    __syncthreads();
    for (int w = 0; w < warp; ++w) {
        a += s.wc[w];
        b += s.ww[w];
    }
}

// fcnt: this CTA's values, two 16-bit counts a word (kFbRange / 2 words).
SV_DEV void fallback_rows(const RowParams& p, uint32_t* fcnt, FallbackShared& s) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31;
    const int V = p.V, nvec = V >> 3;
    const float c2 = p.c2;
    const long long nrows = (long long)p.B * p.rows_per_b;
    (void)nrows;  // bounds of the debug build's checks
    const unsigned nq = __ldcg(p.work + 3);
    const int r0 = rank * kFbRange;  // this CTA's first descending rank
    // local value l of this CTA: descending rank r0 + l, ordinal kFbValues - 1 - (r0 + l)
    const auto count_of = [&](int l) { return (fcnt[l >> 1] >> ((l & 1) * 16)) & 0xFFFFu; };
    for (;;) {
        if (rank == 0 && tid == 0) s.job = (int)atomicAdd(p.work + 4, 1u);
        cl.sync();
        const int qi = *cl.map_shared_rank(&s.job, 0);
        cl.sync();  // every CTA has read the job (rank 0 may now exit or take the next)
        if (qi >= (int)nq) break;  // (the same for every CTA of the cluster)
        const int row = SV_IN(qi, nrows) ? __ldcg(p.fb_rows + qi) : 0;
        RowRec* rec = p.rows + row;
        const float m = __ldcg(&rec->m), S = __ldcg(&rec->S);
        const float mc = m * c2;
        for (int i = tid; i < kFbRange / 8; i += NT) reinterpret_cast<uint4*>(fcnt)[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        const uint4* src = reinterpret_cast<const uint4*>(row_src(p, row / p.rows_per_b, row % p.rows_per_b));
        const auto add = [&](uint32_t raw) {
            const int l = kFbValues - 1 - (int)ord16(raw) - r0;
            if ((unsigned)l < (unsigned)kFbRange) atomicAdd(&fcnt[l >> 1], 1u << ((l & 1) * 16));
        };
#pragma unroll 4
        for (int v = tid; v < nvec; v += NT) {
            const uint4 x = __ldg(src + v);
            add(x.x & 0xFFFFu);
            add(x.x >> 16);
            add(x.y & 0xFFFFu);
            add(x.y >> 16);
            add(x.z & 0xFFFFu);
            add(x.z >> 16);
            add(x.w & 0xFFFFu);
            add(x.w >> 16);
        }
        __syncthreads();
        // this thread's values: totals (each lane starts at its own offset,
        // so a warp's reads fall in different banks), the threads' places in
        // the CTA, then the CTAs' places in the cluster
        const int l0 = tid * kFbPer;
        const auto mass_of = [&](int l, unsigned c) {
            return (unsigned long long)c *
                   fx_of(fmaf(ord16_value((uint32_t)(kFbValues - 1 - (r0 + l))), c2, -mc));
        };
        unsigned long long tc = 0ull, tw = 0ull;
        for (int i = 0; i < kFbPer; ++i) {
            const int l = l0 + ((i + lane) & (kFbPer - 1));
            const unsigned c = count_of(l);
            if (c) {
                tc += c;
                tw += mass_of(l, c);
            }
        }
        unsigned long long ec = tc, ew = tw;
        block_scan2(s, ec, ew);
        if (tid == NT - 1) {
            s.cc = ec;
            s.cw = ew;
        }
        ec -= tc;
        ew -= tw;
        cl.sync();  // every CTA's totals are posted
        for (int q = 0; q < rank; ++q) {
            ec += *cl.map_shared_rank(&s.cc, q);
            ew += *cl.map_shared_rank(&s.cw, q);
        }
        // the first descending rank d <= dlim whose running weight reaches
        // the target, and the mass through it (-1 if none), the same in
        // every CTA of the cluster
        const auto find = [&](bool by_count, unsigned long long target, int dlim, unsigned long long* wo) {
            if (tid == 0) s.hit = -1;
            __syncthreads();
            if ((by_count ? ec : ew) < target && (by_count ? ec + tc : ew + tw) >= target && r0 + l0 <= dlim) {
                unsigned long long c = ec, w = ew;
                for (int l = l0; l < l0 + kFbPer && r0 + l <= dlim; ++l) {
                    const unsigned k = count_of(l);
                    if (!k) continue;
                    c += k;
                    w += mass_of(l, k);
                    if ((by_count ? c : w) >= target) {
                        s.hit = r0 + l;
                        s.hw = w;
                        break;
                    }
                }
            }
            cl.sync();  // every CTA's result is posted
            int d = -1;
            unsigned long long w = 0ull;
            for (int q = 0; q < kFbCluster; ++q) {
                const int h = *cl.map_shared_rank(&s.hit, q);
                if (h >= 0) {
                    d = h;
                    w = *cl.map_shared_rank(&s.hw, q);
                }
            }
            cl.sync();  // every CTA has read the results before they are reset
            *wo = w;
            return d;
        };
        unsigned long long kept = (unsigned long long)(S * kFx);
        float thr = -INFINITY;
        int dk = kFbValues - 1;
        if (p.transform & kXfTopK) {
            unsigned long long w;
            const int d = find(true, (unsigned long long)p.top_k, dk, &w);
            if (d >= 0) {  // (k beyond the row: every logit is kept)
                dk = d;
                thr = ord16_value((uint32_t)(kFbValues - 1 - d));
                kept = w;
            }
        }
        if (p.transform & kXfTopP) {
            unsigned long long w;
            const int d = find(false, top_p_target(p.top_p, kept), dk, &w);
            if (d >= 0) {
                thr = ord16_value((uint32_t)(kFbValues - 1 - d));
                kept = w;
            }
        }
        if (rank == 0 && tid == 0) {
            rec->thr = thr;
            rec->Sk = (float)kept * (1.0f / kFx);
        }
        cl.sync();  // the counts, the shared state and rank 0's job are free for the next row
    }
}

// ---- per sequence: acceptance, then the one draw --------------------------------

// Inverse CDF by one warp over a window list of K entries in order: flat
// position j lies in region r (off[r] <= j < off[r] + cnt[r]) at entry
// e = r kKeptRegionCap + j - off[r] of le, which holds (index << 16) | raw
// target logit; its weight is wf(zt, fetch(entry)), fetch giving the draft
// logit where the weight needs one. The result is the index of the
// smallest j with C_j > u W (C the inclusive prefix sum, W the total), or,
// if rounding leaves none, of the last j with positive weight; -1 when
// W = 0. The positions go in rounds of 32 (lane l takes position 32 s + l
// of round s), kDrawBatch rounds at a time so that their list loads, and
// then their gathers, are in flight together; the first batch stays in
// registers for the second pass, later batches are loaded again. W adds the
// rounds' butterfly totals in round order (the same value in every lane); C
// adds the rounds' scans in round order. Every lane of the warp calls it
// and gets the result.
constexpr int kDrawBatch = 8;

template <typename FETCH, typename WF>
SV_DEV int warp_list_draw(int K, const int* off, const uint32_t* le, float u, const FETCH& fetch, const WF& wf,
                          float* W_out) {
    const int lane = threadIdx.x & 31;
    const int ns = (K + 31) >> 5;
    // weights and entries of rounds s0 .. s0 + kDrawBatch - 1 (0 past K); rg
    // is the lane's region cursor, which only moves forward
    const auto batch = [&](int s0, int& rg, float(&w)[kDrawBatch], uint32_t(&en)[kDrawBatch]) {
        int e[kDrawBatch];
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) {
            const int j = (s0 + q) * 32 + lane;
            e[q] = -1;
            if (j < K) {
                while (rg < kKeptRegions - 1 && off[rg + 1] <= j) ++rg;
                e[q] = rg * kKeptRegionCap + j - off[rg];
            }
        }
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) en[q] = e[q] >= 0 ? __ldg(le + e[q]) : 0u;
        float zd[kDrawBatch];
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) zd[q] = e[q] >= 0 ? fetch(en[q]) : 0.f;
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) w[q] = e[q] >= 0 ? wf(__uint_as_float(en[q] << 16), zd[q]) : 0.f;
    };
    const auto round_total = [](float v) {
        // (lanes l and l ^ o add the same two values, so every lane ends with the same total)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        return v;
    };
    float wk[kDrawBatch];
    uint32_t ek[kDrawBatch];
    int rg = 0;
    batch(0, rg, wk, ek);
    float W = 0.f;
#pragma unroll
    for (int q = 0; q < kDrawBatch; ++q) W += round_total(wk[q]);
    for (int s0 = kDrawBatch; s0 < ns; s0 += kDrawBatch) {
        float w[kDrawBatch];
        uint32_t en[kDrawBatch];
        batch(s0, rg, w, en);
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) W += round_total(w[q]);
    }
    *W_out = W;
    if (!(W > 0.f)) return -1;
    const float t = u * W;
    float base = 0.f;  // C before the round
    int last = -1;     // the index of the last entry with positive weight so far
    // the index at the crossing in a round (the same in every lane), or -1
    const auto cross = [&](float w, uint32_t en) {
        float c = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, c, o);
            if (lane >= o) c += y;
        }
        c += base;
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, w > 0.f && c > t);
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, w > 0.f);
        if (pos) last = (int)(__shfl_sync(0xFFFFFFFFu, en, 31 - __clz(pos)) >> 16);
        base = __shfl_sync(0xFFFFFFFFu, c, 31);
        return hit ? (int)(__shfl_sync(0xFFFFFFFFu, en, __ffs(hit) - 1) >> 16) : -1;
    };
#pragma unroll
    for (int q = 0; q < kDrawBatch; ++q) {
        const int r = cross(wk[q], ek[q]);
        if (r >= 0) return r;
    }
    rg = 0;
    for (int s0 = kDrawBatch; s0 < ns; s0 += kDrawBatch) {
        float w[kDrawBatch];
        uint32_t en[kDrawBatch];
        batch(s0, rg, w, en);
#pragma unroll
        for (int q = 0; q < kDrawBatch; ++q) {
            const int r = cross(w[q], en[q]);
            if (r >= 0) return r;
        }
    }
    return last;
}

// A lane's row record, read by every lane of the warp.
SV_DEV RowRec shfl_rec(const RowRec& r, int src) {
    RowRec o;
    o.m = __shfl_sync(0xFFFFFFFFu, r.m, src);
    o.S = __shfl_sync(0xFFFFFFFFu, r.S, src);
    o.thr = __shfl_sync(0xFFFFFFFFu, r.thr, src);
    o.Sk = __shfl_sync(0xFFFFFFFFu, r.Sk, src);
    o.zx = __shfl_sync(0xFFFFFFFFu, r.zx, src);
    o.x = __shfl_sync(0xFFFFFFFFu, r.x, src);
    o.flags = __shfl_sync(0xFFFFFFFFu, r.flags, src);
    o.nkept = __shfl_sync(0xFFFFFFFFu, r.nkept, src);
    return o;
}

// One warp per sequence (warp w0 + i nwarps takes sequence i ... : the
// caller numbers its warps): the acceptance tests of all positions at once
// (lane k loads target record k and draft record k, 32 positions a round),
// the first rejection n, the accepted prefix, and the draw from the window
// list of target row n, whose record and region sizes the warp already
// holds (the region sizes of every target row of the sequence are loaded
// with the records), so that only the list and the draft logits it names
// are loaded after n is known. A sequence is queued (p.seq_n, counted in
// p.work[0]) for smem_fulldraw_kernel, which resolves it again from the
// rows, when one of its rows takes its threshold from the fallback (which
// may still be running: nothing of the sequence is written here) or when
// its target row n has no usable list (a region of the list overflowed).
// roff: a [NW][kKeptRegions] table in shared memory, one row per warp.
SV_DEV void draw_sequences(const RowParams& p, int (*roff)[kKeptRegions], long long w0, long long nwarps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = p.rows_per_b, G = p.gamma;
    const float c2 = p.c2;
    const int cw = 3 * (G + 1);  // 4-byte words of region sizes of a sequence's target rows
    static_assert(kKeptRegions == 12, "region sizes of a row: three 4-byte words");
    for (long long bb = w0; bb < p.B; bb += nwarps) {
        const int b = (int)bb;
        const RowRec* rb = p.rows + (size_t)b * R;
        const size_t trow0 = (size_t)b * (G + 1);
        const uint32_t* kwp = reinterpret_cast<const uint32_t*>(p.kept_cnt + trow0 * kKeptRegions);
        const uint32_t kw =
            (p.kept_cnt && lane < cw && SV_IN(trow0 * 3 + lane, (long long)p.B * cw)) ? __ldcg(kwp + lane) : 0u;
        // acceptance at every position (lenience l scales the draft
        // probability; l = 1 is the exact method); n = the first rejection,
        // tn and dn its target and draft records
        int flags = 0, n = -1, x0 = -1;
        RowRec tn{}, dn{};
        for (int k0 = 0; k0 <= G; k0 += 32) {
            const int k = k0 + lane;
            RowRec t{}, d{};
            if (k <= G) t = load_rec(rb + k);
            if (k < G) d = load_rec(rb + G + 1 + k);
            bool rej = false;
            if (k < G) {
                const float q = KeptExp{t.thr, c2, t.m * c2, 1.f}(t.zx) / t.Sk;
                const float pd = KeptExp{d.thr, c2, d.m * c2, 1.f}(d.zx) / d.Sk;
                if (p.probs_dbg) {
                    p.probs_dbg[((size_t)b * G + k) * 2 + 0] = q;
                    p.probs_dbg[((size_t)b * G + k) * 2 + 1] = pd;
                }
                const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
                rej = !accept_test(u, q, p.lenience * pd);
            }
            flags |= t.flags | d.flags;
            if (k0 == 0) x0 = t.x;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, rej);
            if (n < 0 && (m || k0 + 32 > G)) {
                n = m ? k0 + __ffs(m) - 1 : G;
                tn = shfl_rec(t, n - k0);
                dn = shfl_rec(d, n - k0);
            }
        }
        flags = __reduce_or_sync(0xFFFFFFFFu, flags);
        if (flags & kRecFallback) {
            if (lane == 0) p.seq_n[atomicAdd(p.work, 1u)] = b;  // resolved from the rows afterwards
            continue;
        }
        const int stt = (flags & kRecTimeout) ? kETimeout : ((flags & kRecEData) ? kEData : kOk);
        if (lane == 0) {
            p.accepted[b] = stt ? -1 : n;
            if (stt) p.next_token[b] = -1;
            if (p.status) p.status[b] = stt;
        }
        for (int j = lane; j <= G; j += 32)
            if ((stt || j != n) && SV_IN_SEQ(trow0 + j, (long long)p.B * (G + 1), p.status, b))
                p.tokens[trow0 + j] = (!stt && j < n) ? (j < 32 ? x0 : __ldcg(&rb[j].x)) : -1;
        if (stt) continue;
        if (tn.nkept < 0 || !SV_IN_SEQ(tn.nkept, p.kept_cap + 1, p.status, b)) {
            if (lane == 0) p.seq_n[atomicAdd(p.work, 1u)] = b;  // drawn from the rows afterwards
            continue;
        }
        // from the window list of target row n (every index with q > 0
        // lies in it; entries below the threshold weigh 0): its region
        // sizes (bytes 12 n .. 12 n + 11 of the sequence's), their offsets
        {
            int c;
            if (cw <= 32) {
                const uint32_t wv = __shfl_sync(0xFFFFFFFFu, kw, min(3 * n + (lane >> 2), 31));
                c = lane < kKeptRegions ? (int)((wv >> ((lane & 3) * 8)) & 0xFFu) : 0;
            } else {
                c = lane < kKeptRegions ? (int)__ldcg(p.kept_cnt + (trow0 + n) * kKeptRegions + lane) : 0;
            }
            int o = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, o, d);
                if (lane >= d) o += y;
            }
            if (lane < kKeptRegions) roff[warp][lane] = o - c;
            __syncwarp();
        }
        const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)n, kPurposeResample);
        // (the list was written by the previous kernel: read-only loads)
        const uint32_t* le = p.kept + (trow0 + n) * (size_t)p.kept_cap;  // (index << 16) | raw
        const RowRec& t = tn;
        const KeptExp q1{t.thr, c2, t.m * c2, 1.f};
        const auto no_draft = [](uint32_t) { return 0.f; };
        const auto wq = [&](float zt, float) { return q1(zt); };
        float W = 0.f;
        int tok = -1;
        if (n < G) {
            const unsigned short* rd = reinterpret_cast<const unsigned short*>(p.draft) + ((size_t)b * G + n) * p.V;
            const ResidualW rw = residual_weight(t, dn, c2, p.lenience);
            const auto draft_of = [&](uint32_t en) {
                if (!(__uint_as_float(en << 16) >= t.thr)) return 0.f;  // q = 0: the draft logit is not needed
                const uint32_t i = en >> 16;
                return SV_IN_SEQ(i, p.V, p.status, b) ? __uint_as_float((uint32_t)__ldg(rd + i) << 16) : 0.f;
            };
            const auto wr = [&](float zt, float zd) { return zt >= t.thr ? rw(zt, zd) : 0.f; };
            tok = warp_list_draw(t.nkept, roff[warp], le, u2, draft_of, wr, &W);
        }
        if (!(W > 0.f)) tok = warp_list_draw(t.nkept, roff[warp], le, u2, no_draft, wq, &W);  // bonus, or a vanished residual
        __syncwarp();  // the region table is read before the warp's next sequence rewrites it
        if (lane == 0) {
            p.next_token[b] = tok;
            p.tokens[trow0 + n] = tok;
        }
    }
}

// After the row kernel: the queued rows' thresholds and every sequence's
// acceptance and draw in one launch. The first fb_ctas CTAs (whole
// clusters) take the queued rows (fallback_rows), the warps of the others
// take the sequences (draw_sequences); a sequence with a queued row is left
// to smem_fulldraw_kernel, which runs once every record is complete, so no
// CTA waits for one outside its own cluster.
__global__ void __cluster_dims__(kFbCluster, 1, 1) __launch_bounds__(NT, 4)
    smem_tail_kernel(const __grid_constant__ RowParams p, const int fb_ctas) {
    __shared__ uint32_t fcnt[kFbRange / 2];
    __shared__ FallbackShared s;
    __shared__ int roff[NW][kKeptRegions];
    if ((int)blockIdx.x < fb_ctas) {
        fallback_rows(p, fcnt, s);  // (fb_ctas is a multiple of the cluster size: whole clusters)
        return;
    }
    draw_sequences(p, roff, (long long)(blockIdx.x - fb_ctas) * NW + (threadIdx.x >> 5),
                   (long long)(gridDim.x - fb_ctas) * NW);
}

// The queued sequences: one CTA per sequence resolves it from its records,
// all complete by now (acceptance at every position, one thread each; the
// first rejection n; the accepted prefix), then draws from the residual row
// pair, or the bonus row, in global memory with the CTA-wide inverse CDF of
// draw.cuh, four 16-byte vectors of each row per thread and round in flight
// (a 32000-logit row is four rounds). The acceptance arithmetic is
// draw_sequences' own, so a sequence it queued after writing its outputs
// (no usable list) gets the same n and prefix again.
constexpr int kFullVec = 4;
__global__ void __launch_bounds__(NT) smem_fulldraw_kernel(const __grid_constant__ RowParams p) {
    __shared__ DrawShared ds;
    __shared__ int job, sn, sfl;
    const int tid = threadIdx.x;
    const int R = p.rows_per_b, G = p.gamma, V = p.V;
    const float c2 = p.c2;
    const unsigned nq = __ldcg(p.work);
    for (;;) {
        if (tid == 0) {
            job = (int)atomicAdd(p.work + 2, 1u);
            sn = G;
            sfl = 0;
        }
        __syncthreads();
        const int qi = job;
        if (qi >= (int)nq) break;
        const int b = SV_IN(qi, p.B) ? __ldcg(p.seq_n + qi) : 0;
        const RowRec* rb = p.rows + (size_t)b * R;
        int fl = 0;
        for (int i = tid; i < R; i += NT) fl |= __ldcg(&rb[i].flags);
        if (fl) atomicOr(&sfl, fl);
        for (int k = tid; k < G; k += NT) {
            const RowRec t = load_rec(rb + k), d = load_rec(rb + G + 1 + k);
            const float q = KeptExp{t.thr, c2, t.m * c2, 1.f}(t.zx) / t.Sk;
            const float pd = KeptExp{d.thr, c2, d.m * c2, 1.f}(d.zx) / d.Sk;
            if (p.probs_dbg) {
                p.probs_dbg[((size_t)b * G + k) * 2 + 0] = q;
                p.probs_dbg[((size_t)b * G + k) * 2 + 1] = pd;
            }
            const float u = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)k, kPurposeAccept);
            if (!accept_test(u, q, p.lenience * pd)) atomicMin(&sn, k);
        }
        __syncthreads();
        const int n = sn, flags = sfl;
        const int stt = (flags & kRecTimeout) ? kETimeout : ((flags & kRecEData) ? kEData : kOk);
        if (tid == 0) {
            p.accepted[b] = stt ? -1 : n;
            if (stt) p.next_token[b] = -1;
            if (p.status) p.status[b] = stt;
        }
        for (int j = tid; j <= G; j += NT)
            if ((stt || j != n) && SV_IN_SEQ((size_t)b * (G + 1) + j, (long long)p.B * (G + 1), p.status, b))
                p.tokens[(size_t)b * (G + 1) + j] = (!stt && j < n) ? __ldcg(&rb[j].x) : -1;
        if (!stt) {  // (the same in every thread)
            const RowRec t = load_rec(rb + n);
            const float u2 = uniform01(p.seed, p.offset + (uint64_t)b, (uint32_t)n, kPurposeResample);
            const bf16_t* rt = reinterpret_cast<const bf16_t*>(p.target) + ((size_t)b * (G + 1) + n) * V;
            int tok;
            if (n < G) {
                const RowRec d = load_rec(rb + G + 1 + n);
                const bf16_t* rd = reinterpret_cast<const bf16_t*>(p.draft) + ((size_t)b * G + n) * V;
                tok = draw_residual<bf16_t, kFullVec>(ds, rt, rd, V, t, d, c2, u2, p.lenience);
            } else {
                tok = draw_q<bf16_t, kFullVec>(ds, rt, V, t, c2, u2);
            }
            if (tid == 0) {
                p.next_token[b] = tok;
                p.tokens[(size_t)b * (G + 1) + n] = tok;
            }
        }
        __syncthreads();  // job, sn and sfl are read before thread 0 resets them
    }
}

}  // namespace

bool smem_rows_plan(int V, int* nbuf, size_t* smem) {
    if (V < 8 || V > 65536 || (V & 7)) return false;
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, smem_row_kernel) != cudaSuccess)
        return false;
    const size_t rb = ((size_t)V * 2 + 127) & ~(size_t)127;
    const size_t per = rb + kSlotBytes;
    const size_t lists = kListBytes;
    const size_t avail = (size_t)optin > fa.sharedSizeBytes + lists ? (size_t)optin - fa.sharedSizeBytes - lists : 0;
    const int n = (int)std::min<size_t>(kMaxSlots, avail / per);
    if (n < 2) return false;  // a ring of at least two rows
    *nbuf = n;
    *smem = (size_t)n * per + lists;
    return true;
}

cudaError_t launch_smem_rows(const RowParams& p, int nbuf, size_t smem, int sms, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(smem_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.rows_per_b;
    const int grid = (int)(rows < sms ? rows : sms);
    smem_row_kernel<<<grid, kRowThreads, smem, stream>>>(p, nbuf);
    return cudaGetLastError();
}

cudaError_t launch_smem_draws(const RowParams& p, int sms, cudaStream_t stream) {
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, smem_tail_kernel, NT, 0) != cudaSuccess || n < 1) n = 1;
        return n;
    }();
    // the queued rows (usually a few: the other clusters find the queue
    // empty and exit at once), then the sequences' warps, whole clusters
    const int fb_ctas = std::max(1, sms / kFbCluster) * kFbCluster;
    long long dr = std::min<long long>(((long long)p.B + NW - 1) / NW, (long long)sms * per_sm);
    dr = (dr + kFbCluster - 1) / kFbCluster * kFbCluster;
    smem_tail_kernel<<<(unsigned)(fb_ctas + dr), NT, 0, stream>>>(p, fb_ctas);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the queued sequences (usually a few; CTAs that find the queue empty exit)
    smem_fulldraw_kernel<<<sms, NT, 0, stream>>>(p);
    return cudaGetLastError();
}

SV_DEBUG_READER(rows_smem)

}  // namespace sv

extern "C" int spec_debug_withhold_copy(int j) {
#ifdef SPEC_DEBUG
    return cudaMemcpyToSymbol(sv::g_withhold, &j, sizeof(int)) == cudaSuccess ? 0 : -1;
#else
    (void)j;
    return -1;
#endif
}
