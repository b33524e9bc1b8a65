// Shared device helpers and launch parameter blocks for libspecverify.
//
// Everything here is GB300 (sm_103a) device code or plain host structs; the
// CPU oracle in the repository does not include or call any of it.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#define SV_DEV __device__ __forceinline__
#define SV_HD __host__ __device__ __forceinline__

namespace sv {

// Status codes written to status[b] (mirror spec_status in specverify.h).
constexpr int kOk = 0;
constexpr int kEData = 4;
constexpr int kETimeout = 3;

// ---------------------------------------------------------------------------
// Index checks of the debug build (-DSPEC_DEBUG, build.py's debug library).
// SV_IN(i, n) checks 0 <= i < n for an index a kernel is about to use; a
// failed check counts the failure in the translation unit's failure words,
// keeps the source line of the first one, and returns false so that the
// caller skips the access (nothing traps or faults). SV_IN_SEQ also marks the
// sequence's status with kEBounds. Release builds compile both to `true`.
// Each translation unit keeps its own words (the library is built without
// relocatable device code) and reads them with SV_DEBUG_READER.
// ---------------------------------------------------------------------------
constexpr int kEBounds = 5;

#ifdef SPEC_DEBUG
static __device__ unsigned int g_sv_debug[2];  // failed checks, line of the first

SV_DEV bool sv_in(long long i, long long n, int line) {
    if (i >= 0 && i < n) return true;
    if (atomicAdd(&g_sv_debug[0], 1u) == 0u) g_sv_debug[1] = (unsigned)line;
    return false;
}

SV_DEV bool sv_in_seq(long long i, long long n, int line, int32_t* status, long long b) {
    if (sv_in(i, n, line)) return true;
    if (status) atomicMax(reinterpret_cast<int*>(status + b), kEBounds);
    return false;
}

#define SV_IN(i, n) ::sv::sv_in((long long)(i), (long long)(n), __LINE__)
#define SV_IN_SEQ(i, n, status, b) ::sv::sv_in_seq((long long)(i), (long long)(n), __LINE__, (status), (long long)(b))
// Defines sv::debug_read_<tu>(count, line): this translation unit's words.
#define SV_DEBUG_READER(tu)                                                        \
    cudaError_t debug_read_##tu(unsigned int* count, unsigned int* line) {        \
        unsigned int w[2] = {0u, 0u};                                             \
        const cudaError_t e = cudaMemcpyFromSymbol(w, g_sv_debug, sizeof(w));     \
        *count = w[0];                                                            \
        *line = w[1];                                                             \
        return e;                                                                 \
    }
#else
#define SV_IN(i, n) true
#define SV_IN_SEQ(i, n, status, b) true
#define SV_DEBUG_READER(tu)                                                        \
    cudaError_t debug_read_##tu(unsigned int* count, unsigned int* line) {        \
        *count = 0u;                                                              \
        *line = 0u;                                                               \
        return cudaSuccess;                                                       \
    }
#endif

// The debug readers of the kernel translation units.
cudaError_t debug_read_rows(unsigned int* count, unsigned int* line);
cudaError_t debug_read_rows_smem(unsigned int* count, unsigned int* line);
cudaError_t debug_read_argmax(unsigned int* count, unsigned int* line);
cudaError_t debug_read_mentor(unsigned int* count, unsigned int* line);
cudaError_t debug_read_beta(unsigned int* count, unsigned int* line);
cudaError_t debug_read_tree_build(unsigned int* count, unsigned int* line);

// Per-task record flags.
constexpr int kRecEData = 2;     // bad logits in this row, or a draft token out of range
constexpr int kRecTimeout = 4;   // the row's staging copy did not complete in time
constexpr int kRecFallback = 8;  // shared-memory path: the row's threshold comes from the fallback selection

constexpr uint32_t kPurposeAccept = 0;
constexpr uint32_t kPurposeResample = 1;

// ---------------------------------------------------------------------------
// Philox-4x32-10, written from Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3" (SC'11). One round maps (c0, c1, c2, c3) to
// (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key
// advances by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
struct Philox4 {
    uint32_t v[4];
};

SV_HD Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                            uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
#ifdef __CUDA_ARCH__
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
#else
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
#endif
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return Philox4{{c0, c1, c2, c3}};
}

// u = ((w0 >> 9) + 0.5) * 2^-23 for counter (row lo, row hi, position, purpose)
// and key (seed lo, seed hi): 2^23 equally likely values in (0, 1), exact in fp32.
SV_HD float uniform01(uint64_t seed, uint64_t row, uint32_t pos, uint32_t purpose) {
    const Philox4 r = philox4x32_10((uint32_t)row, (uint32_t)(row >> 32), pos, purpose,
                                    (uint32_t)seed, (uint32_t)(seed >> 32));
    return ((float)(r.v[0] >> 9) + 0.5f) * 0x1p-23f;
}

// ---------------------------------------------------------------------------
// Order-preserving 32-bit keys of fp32 values (-0 folded onto +0 so that
// equal values share a key). bf16 values converted to fp32 exactly keep all
// their information in the top 16 key bits.
// ---------------------------------------------------------------------------
SV_HD uint32_t f32_key(float x) {
#ifdef __CUDA_ARCH__
    uint32_t b = __float_as_uint(x);
#else
    uint32_t b;
    __builtin_memcpy(&b, &x, 4);
#endif
    b = (b == 0x80000000u) ? 0u : b;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

SV_DEV float key_to_f32(uint32_t k) {
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // f32_key(-inf)
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // f32_key(+inf)

// 2^x on the MUFU unit (ex2.approx.ftz: about 2 ulp).
SV_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// 16-byte vectors of logits.
// ---------------------------------------------------------------------------
template <typename E>
struct VecTraits;

template <>
struct VecTraits<float> {
    static constexpr int kN = 4;
    static constexpr uint32_t kNegInfBits = 0xFF800000u;
    SV_DEV static void unpack(const uint4& r, float (&x)[4]) {
        x[0] = __uint_as_float(r.x);
        x[1] = __uint_as_float(r.y);
        x[2] = __uint_as_float(r.z);
        x[3] = __uint_as_float(r.w);
    }
    SV_DEV static float load1(const void* p) { return __ldg(reinterpret_cast<const float*>(p)); }
};

struct bf16_t {
    uint16_t bits;
};

template <>
struct VecTraits<bf16_t> {
    static constexpr int kN = 8;
    static constexpr uint32_t kNegInfBits = 0xFF80u;
    SV_DEV static void unpack(const uint4& r, float (&x)[8]) {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xFFFF0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        x[4] = __uint_as_float(r.z << 16);
        x[5] = __uint_as_float(r.z & 0xFFFF0000u);
        x[6] = __uint_as_float(r.w << 16);
        x[7] = __uint_as_float(r.w & 0xFFFF0000u);
    }
    SV_DEV static float load1(const void* p) {
        const unsigned short v = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(((uint32_t)v) << 16);
    }
};

// Streaming 16-byte global load: read once, do not keep in L1.
SV_DEV uint4 ld_stream_v4(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// Warp reductions.
// ---------------------------------------------------------------------------
SV_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
SV_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
SV_DEV unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
}
SV_DEV uint32_t warp_min_u32(uint32_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Exclusive prefix of v over lanes 0..31 in lane order, summed sequentially so
// that prefix[l+1] == prefix[l] + v[l] exactly. Returns the lane's exclusive
// prefix; *total receives the sequential total.
SV_DEV float warp_seq_exclusive(float v, float* total) {
    const int lane = threadIdx.x & 31;
    float acc = 0.f, mine = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        if (j == lane) mine = acc;
        acc += __shfl_sync(0xFFFFFFFFu, v, j);
    }
    *total = acc;
    return mine;
}

// ---------------------------------------------------------------------------
// Launch parameter blocks (host and device).
// ---------------------------------------------------------------------------
enum RowMode : int { kModeVerify = 0, kModeMentor = 1, kModeSample = 2 };
enum Transform : int { kXfTopK = 1, kXfTopP = 2 };

// One record per logit row (workspace), written by the CTA that completes the row.
struct alignas(16) RowRec {
    float m;      // row maximum
    float S;      // sum of exp2((z - m) log2e / T) over the row
    float thr;    // kept set: z >= thr (-inf: the whole row)
    float Sk;     // kept mass (the normaliser of the row's probabilities)
    float zx;     // the draft token's logit in this row (rows with a token)
    int32_t x;    // the draft token (rows with a token), else -1
    int32_t flags;  // kRecEData, kRecTimeout, kRecFallback
    int32_t nkept;  // shared-memory row path, target rows: entries of the window list (-1: none)
};

// Partial statistics of one segment of a long row.
struct SegRec {
    float m, s, zx;
    int32_t flags;
};

// Window lists of the shared-memory row path (see RowParams::kept_idx).
constexpr int kKeptRegions = 12;
constexpr int kKeptRegionCap = 128;

struct RowParams {
    const void* target;
    const void* draft;
    const int32_t* draft_tokens;
    int B, gamma, V;
    int rows_per_b;   // 2 gamma + 1 (verify / mentor) or P (sample)
    int nseg;         // segments per row
    int seg_len;      // elements per segment (multiple of 16)
    int mode;         // RowMode
    int transform;    // Transform bits
    int top_k;
    float top_p;
    float c2;         // log2(e) / T
    float lenience;   // l in ]0, 1]: the draft probability is scaled by l (1: exact)
    uint64_t seed, offset;
    uint32_t pos0, purpose;  // sample mode
    int32_t* accepted;
    int32_t* tokens;
    int32_t* next_token;
    int32_t* status;
    float* probs_dbg;
    int32_t* sample_out;
    RowRec* rows;           // [B * rows_per_b]
    SegRec* segs;           // [B * rows_per_b * nseg] (nseg > 1)
    unsigned int* row_cnt;  // [B * rows_per_b] segment arrivals (nseg > 1)
    unsigned int* seq_cnt;  // [B] row arrivals
    unsigned int* work;     // work counters (zero at launch): [0] next work unit (row kernel) or
                            // queued sequences, [1] next sequence to draw (streaming path),
                            // [2] next queued sequence, [3] queued rows, [4] next queued row
    int32_t* seq_n;         // [B] accepted length of each resolved sequence (-1: bad data)
    // shared-memory row path: the window list of every target row (the
    // logits within the window of its maximum, a superset of its kept set):
    // kKeptRegions regions of kKeptRegionCap entries (index << 16 | raw bf16),
    // each region in ascending index order, the regions in order; kept_cnt
    // holds the entries of each region
    uint32_t* kept;         // [B * (gamma + 1) * kept_cap]
    uint8_t* kept_cnt;      // [B * (gamma + 1) * kKeptRegions]
    int kept_cap;           // kKeptRegions * kKeptRegionCap
    int32_t* fb_rows;       // [B * rows_per_b] rows whose threshold comes from the whole row
};

enum ArgmaxMode : int { kArgVerify = 0, kArgTree = 1, kArgSample = 2 };

struct ArgmaxParams {
    const void* logits;
    int B, rows_per_b, V;
    int mode;          // ArgmaxMode
    int chunk;         // elements per CTA (flattened [rows, V] range)
    int max_depth;     // tree
    const int32_t* draft_tokens;  // verify: [B, rows_per_b - 1]
    const int32_t* node_tokens;   // tree: [B, N]
    const int32_t* parent;
    const int32_t* depth;
    int32_t* out0;  // verify: accepted; tree: accept_len; sample: tokens_out
    int32_t* out1;  // verify: tokens;   tree: path_nodes
    int32_t* out2;  // verify: next;     tree: tokens
    int32_t* out3;  // tree: bonus
    float* probs_dbg;  // verify: [B, gamma, 2] (q(x), p(x)) of greedy verification
    int32_t* status;
    unsigned long long* rowbest;  // [rows] packed (key << 32) | ~index
    unsigned int* rowbad;         // [rows]
    unsigned long long* cnt;      // [B] elements processed
};

struct MentorParams {
    const void* target;
    const void* draft;
    int B, gamma, V;
    int bf16;             // logits are bf16 (else fp32)
    float c2;             // log2(e) / T
    float inv_t;          // 1 / T
    float kl_bound;
    int iters;
    uint64_t seed, offset;
    const RowRec* rows;   // from the row kernel (mentor mode)
    uint32_t* keys;       // scratch per slot: [2][V] keys
    uint32_t* idx;        // scratch per slot: [2][V] indices
    float* arr;           // scratch per slot: [7][V] sorted arrays
    unsigned int* work;   // next (sequence, position) job (zero at launch)
    unsigned int* rejmark;  // [B]: max over rejected positions k of gamma - k (zero at launch)
    int32_t* pos_state;   // [B, gamma]: outcome of each solved position
    float* pos_beta;      // [B, gamma]: beta of each solved position
    float* pos_scale;     // [B, gamma, 2]: the solve's normalised 1/S_t and 1/S_d
    int32_t* accepted;
    int32_t* tokens;
    int32_t* next_token;
    int32_t* status;
    float* alpha_out;
    float* beta_out;
    float* probs_dbg;
};

// Host launchers (defined in the .cu files).
// Persistent row kernel on up to `sms` x (resident CTAs per SM) CTAs.
cudaError_t launch_rows(const RowParams& p, int dtype, int sms, cudaStream_t stream);
// The one draw of every sequence the row kernel resolved (verification).
cudaError_t launch_draws(const RowParams& p, int dtype, int sms, cudaStream_t stream);
// Shared-memory row path (bf16 rows with a top-k / top-p transform):
// whether a shape can take it (and the ring depth and dynamic shared memory
// it needs), the row kernel, and the per-sequence resolve and draw.
bool smem_rows_plan(int V, int* nbuf, size_t* smem);
cudaError_t launch_smem_rows(const RowParams& p, int nbuf, size_t smem, int sms, cudaStream_t stream);
cudaError_t launch_smem_draws(const RowParams& p, int sms, cudaStream_t stream);
// Resident argmax CTAs per SM (occupancy of the kernel as built).
int argmax_ctas_per_sm(int dtype);
cudaError_t launch_argmax(const ArgmaxParams& p, int dtype, int grid, cudaStream_t stream);
// Position kernel on `grid` persistent CTAs, then the per-sequence resolve.
cudaError_t launch_mentor(const MentorParams& p, int grid, int resolve_grid, cudaStream_t stream);
// beta[b, k] = sum_x min(q(x), p(x)) of every target / draft row pair, from
// the row records (persistent CTAs over the B * gamma pairs).
cudaError_t launch_beta(const RowParams& p, int dtype, float* beta, int sms, cudaStream_t stream);
// REST draft-tree construction: one CTA per sequence.
size_t tree_build_smem_bytes();
cudaError_t launch_tree_build(const int32_t* cand, const int32_t* counts, const int32_t* root, int B, int C,
                              int L, int V, int N, int32_t* tokens, int32_t* parent, int32_t* depth,
                              uint8_t* mask, int32_t* n_nodes, int32_t* status, cudaStream_t stream);

}  // namespace sv
