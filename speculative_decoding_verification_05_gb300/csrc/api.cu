// C ABI of libspecverify: argument validation, workspace layout, launch
// configuration. Every entry point checks its arguments on the host before
// touching CUDA, so invalid calls return SPEC_EINVAL with nothing enqueued.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "specverify.h"

namespace sv {
spec_status note_cuda_error(cudaError_t e);
}

namespace {

thread_local char g_cuda_err[256] = "";

constexpr size_t kAlign = 256;

size_t al(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

spec_status cuda_fail(cudaError_t e) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return SPEC_ECUDA;
}

int device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        cache[dev] = v;
    }
    return cache[dev];
}

bool finite(float x) { return std::isfinite(x); }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int esize(spec_dtype d) { return d == SPEC_F32 ? 4 : 2; }

bool dtype_ok(spec_dtype d) { return d == SPEC_F32 || d == SPEC_BF16; }

// ---- workspace layouts -----------------------------------------------------

// Segments per row for the row kernel: long rows are split so that a step
// has about kUnitsWanted work units (dynamic scheduling then balances the SMs),
// each at least kMinSeg elements and a multiple of 16 elements. Rows with a
// top-k / top-p transform stay whole (their threshold comes from the whole
// row in one CTA). Depends only on the shape, so results do not depend on the
// device's SM count.
constexpr long long kUnitsWanted = 4096;
constexpr int kMinSeg = 4096;

void seg_plan(long long rows, int V, bool xf, int* nseg, int* seg_len) {
    long long n = 1;
    if (!xf) n = std::max(1LL, std::min((kUnitsWanted + rows - 1) / rows, (long long)(V / kMinSeg)));
    long long len = ((V + n - 1) / n + 15) & ~15LL;
    *seg_len = (int)len;
    *nseg = (int)((V + len - 1) / len);
}

// Every layout starts with the control region that must be zero when the
// kernels start (work counters, arrival counters, packed per-row argmaxes);
// each call clears the part it uses with one memset, so the workspace may
// hold anything on entry. Records and scratch follow and are always written
// before they are read.
struct Ws {
    size_t work, seq_cnt, row_cnt, row_zero_end;  // row kernel control
    size_t cnt64, rowbest, rowbad, arg_end;         // argmax control
    size_t rows, segs, seqn, total;
    int nseg_max;
};

Ws ws_layout(int B, int R, int V) {
    Ws w;
    size_t o = 0;
    const size_t rows = (size_t)B * R;
    int seg_len;
    seg_plan((long long)rows, V, false, &w.nseg_max, &seg_len);
    w.work = o;
    o = al(o + 2 * sizeof(unsigned int));
    w.seq_cnt = o;
    o = al(o + (size_t)B * sizeof(unsigned int));
    w.row_cnt = o;
    o = al(o + rows * sizeof(unsigned int));
    w.row_zero_end = o;
    w.cnt64 = o;
    o = al(o + (size_t)B * sizeof(unsigned long long));
    w.rowbest = o;
    o = al(o + rows * sizeof(unsigned long long));
    w.rowbad = o;
    o = al(o + rows * sizeof(unsigned int));
    w.arg_end = o;
    w.rows = o;
    o = al(o + rows * sizeof(sv::RowRec));
    w.segs = o;
    if (w.nseg_max > 1) o = al(o + rows * w.nseg_max * sizeof(sv::SegRec));
    w.seqn = o;
    o = al(o + (size_t)B * sizeof(int32_t));
    w.total = o;
    return w;
}

// Verification workspace: the row layout, plus (for shapes the shared-memory
// row path can take: bf16, V a multiple of 8, V <= 65536) the window list of
// every target row, kKeptCap entries in regions (index and raw logit packed
// in 32 bits; entries per region), and the queue of rows whose threshold the
// window did not decide.
constexpr int kKeptCap = sv::kKeptRegions * sv::kKeptRegionCap;

struct VerifyWs {
    Ws lin;
    size_t kidx, kcnt, fbq, total;
    bool kept;
};

bool smem_shape(spec_dtype dtype, int V) { return dtype == SPEC_BF16 && V % 8 == 0 && V <= 65536; }

VerifyWs verify_ws(int B, int gamma, int V, spec_dtype dtype) {
    VerifyWs w;
    w.lin = ws_layout(B, 2 * gamma + 1, V);
    size_t o = w.lin.total;
    w.kept = smem_shape(dtype, V);
    w.kidx = w.kcnt = w.fbq = o;
    if (w.kept) {
        const size_t n = (size_t)B * (gamma + 1) * kKeptCap;
        w.kidx = o;
        o = al(o + n * sizeof(uint32_t));
        w.kcnt = o;
        o = al(o + (size_t)B * (gamma + 1) * sv::kKeptRegions);
        w.fbq = o;
        o = al(o + (size_t)B * (2 * gamma + 1) * sizeof(int32_t));
    }
    w.total = o;
    return w;
}

spec_status clear(void* ws, size_t from, size_t to, cudaStream_t st) {
    const cudaError_t e = cudaMemsetAsync(reinterpret_cast<char*>(ws) + from, 0, to - from, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

constexpr int kMentorSlots = 152;

struct MentorWs {
    Ws lin;
    size_t keys, idx, arr, pos_state, pos_beta, pos_scale, total;
    int slots;
};

MentorWs mentor_ws(int B, int gamma, int V) {
    MentorWs w;
    w.lin = ws_layout(B, 2 * gamma + 1, V);
    size_t o = w.lin.total;
    w.slots = (int)std::min<long long>((long long)B * gamma, kMentorSlots);
    w.keys = o;
    o = al(o + (size_t)w.slots * 2 * V * 4);
    w.idx = o;
    o = al(o + (size_t)w.slots * 2 * V * 4);
    w.arr = o;
    o = al(o + (size_t)w.slots * 7 * V * 4);
    w.pos_state = o;
    o = al(o + (size_t)B * gamma * 4);
    w.pos_beta = o;
    o = al(o + (size_t)B * gamma * 4);
    w.pos_scale = o;
    o = al(o + (size_t)B * gamma * 8);
    w.total = o;
    return w;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

// ---- launch configuration ---------------------------------------------------

// Fills the row kernel's workspace pointers and segment plan, clears its
// control region and launches it.
spec_status run_rows(sv::RowParams& p, int dtype, void* ws, const Ws& w, cudaStream_t st) {
    seg_plan((long long)p.B * p.rows_per_b, p.V, p.transform != 0, &p.nseg, &p.seg_len);
    if (p.nseg > w.nseg_max) return SPEC_EINVAL;
    p.rows = at<sv::RowRec>(ws, w.rows);
    p.segs = at<sv::SegRec>(ws, w.segs);
    p.row_cnt = at<unsigned int>(ws, w.row_cnt);
    p.seq_cnt = at<unsigned int>(ws, w.seq_cnt);
    p.work = at<unsigned int>(ws, w.work);
    p.seq_n = at<int32_t>(ws, w.seqn);
    if (spec_status c = clear(ws, 0, w.row_zero_end, st)) return c;
    cudaError_t e = sv::launch_rows(p, dtype, device_sms(), st);
    if (e == cudaSuccess && p.mode == sv::kModeVerify) e = sv::launch_draws(p, dtype, device_sms(), st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

// The shared-memory row path for verification with a transform on bf16
// rows, when the shape, the alignment and the shared memory allow it;
// SPEC_EINVAL (nothing enqueued) when it does not apply.
spec_status run_smem_rows(sv::RowParams& p, void* ws, const VerifyWs& w, cudaStream_t st) {
    int nbuf = 0;
    size_t smem = 0;
    if (!w.kept || p.transform == 0 || p.mode != sv::kModeVerify || !aligned(p.target, 16) ||
        !aligned(p.draft, 16) || (long long)p.B * p.rows_per_b > (1LL << 30) ||
        !sv::smem_rows_plan(p.V, &nbuf, &smem))
        return SPEC_EINVAL;
    p.nseg = 1;
    p.seg_len = p.V;
    p.rows = at<sv::RowRec>(ws, w.lin.rows);
    p.work = at<unsigned int>(ws, w.lin.work);
    p.seq_n = at<int32_t>(ws, w.lin.seqn);  // the queue of sequences drawn from the rows
    p.kept = at<uint32_t>(ws, w.kidx);
    p.kept_cnt = at<uint8_t>(ws, w.kcnt);
    p.kept_cap = kKeptCap;
    p.fb_rows = at<int32_t>(ws, w.fbq);
    if (spec_status c = clear(ws, 0, w.lin.work + kAlign, st)) return c;
    cudaError_t e = sv::launch_smem_rows(p, nbuf, smem, device_sms(), st);
    if (e == cudaSuccess) e = sv::launch_smem_draws(p, device_sms(), st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

spec_status launch_argmax_checked(sv::ArgmaxParams& p, int dtype, void* ws, const Ws& w, cudaStream_t st) {
    p.rowbest = at<unsigned long long>(ws, w.rowbest);
    p.rowbad = at<unsigned int>(ws, w.rowbad);
    p.cnt = at<unsigned long long>(ws, w.cnt64);
    if (spec_status c = clear(ws, w.cnt64, w.arg_end, st)) return c;
    const long long total = (long long)p.B * p.rows_per_b * p.V;
    long long grid = std::min<long long>((long long)device_sms() * sv::argmax_ctas_per_sm(dtype), (total + 8191) / 8192);
    if (grid < 1) grid = 1;
    long long chunk = (total + grid - 1) / grid;
    chunk = (chunk + 63) & ~63LL;
    grid = (total + chunk - 1) / chunk;
    if (chunk > 0x7FFFFFFFLL) return SPEC_EINVAL;
    p.chunk = (int)chunk;
    const cudaError_t e = sv::launch_argmax(p, dtype, (int)grid, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

bool sampling_ok(const spec_sampling& s) {
    return finite(s.temperature) && s.temperature >= 0.f && s.top_p > 0.f && s.top_p <= 1.f &&
           s.top_k >= 0;
}

int transform_bits(const spec_sampling& s, int V) {
    int t = 0;
    if (s.top_k > 0 && s.top_k < V) t |= sv::kXfTopK;
    if (s.top_p < 1.f) t |= sv::kXfTopP;
    return t;
}

const float kLog2e = 1.4426950408889634f;

__global__ void philox_uniform_kernel(uint64_t seed, uint64_t row0, uint32_t pos, uint32_t purpose,
                                      int n, float* out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = sv::uniform01(seed, row0 + (uint64_t)i, pos, purpose);
}

spec_status verify_impl(const void* target, const void* draft, spec_dtype dtype,
                        const int32_t* draft_tokens, int B, int gamma, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset,
                        int32_t* accepted, int32_t* tokens, int32_t* next_token,
                        int32_t* status, float* probs_dbg,
                        void* workspace, size_t ws_bytes, spec_stream stream, float lenience) {
    if (!dtype_ok(dtype) || !sampling_ok(sampling)) return SPEC_EINVAL;
    if (!finite(lenience) || !(lenience > 0.f) || lenience > 1.f) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V)
        return SPEC_EINVAL;
    const bool greedy = sampling.temperature == 0.f;
    if (!target || (!greedy && !draft) || !draft_tokens || !accepted || !tokens || !next_token || !workspace)
        return SPEC_EINVAL;
    const int es = esize(dtype);
    if (!aligned(target, es) || (draft && !aligned(draft, es)) || !aligned(workspace, kAlign))
        return SPEC_EINVAL;
    const VerifyWs vw = verify_ws(B, gamma, V, dtype);
    const Ws& w = vw.lin;
    if (ws_bytes < vw.total) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int dt = dtype == SPEC_F32 ? 0 : 1;

    if (greedy) {
        sv::ArgmaxParams p = {};
        p.logits = target;
        p.B = B;
        p.rows_per_b = gamma + 1;
        p.V = V;
        p.mode = sv::kArgVerify;
        p.draft_tokens = draft_tokens;
        p.out0 = accepted;
        p.out1 = tokens;
        p.out2 = next_token;
        p.probs_dbg = probs_dbg;
        p.status = status;
        return launch_argmax_checked(p, dt, workspace, w, st);
    }
    sv::RowParams p = {};
    p.target = target;
    p.draft = draft;
    p.draft_tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.rows_per_b = 2 * gamma + 1;
    p.mode = sv::kModeVerify;
    p.transform = transform_bits(sampling, V);
    p.top_k = sampling.top_k;
    p.top_p = sampling.top_p;
    p.c2 = kLog2e / sampling.temperature;
    p.lenience = lenience;
    p.seed = seed;
    p.offset = offset;
    p.accepted = accepted;
    p.tokens = tokens;
    p.next_token = next_token;
    p.status = status;
    p.probs_dbg = probs_dbg;
    if (!std::isfinite(p.c2)) return SPEC_EINVAL;
    if (dt == 1 && p.transform != 0) {
        const spec_status s = run_smem_rows(p, workspace, vw, st);
        if (s != SPEC_EINVAL) return s;
    }
    return run_rows(p, dt, workspace, w, st);
}

}  // namespace

// Records a CUDA error for spec_last_cuda_error (used by other translation units).
spec_status sv::note_cuda_error(cudaError_t e) { return cuda_fail(e); }

extern "C" {

int spec_version(void) { return 100; }

const char* spec_status_string(spec_status s) {
    switch (s) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_EINVAL: return "SPEC_EINVAL";
        case SPEC_ECUDA: return "SPEC_ECUDA";
        case SPEC_ETIMEOUT: return "SPEC_ETIMEOUT";
        case SPEC_EDATA: return "SPEC_EDATA";
        case SPEC_EBOUNDS: return "SPEC_EBOUNDS";
    }
    return "SPEC_UNKNOWN";
}

const char* spec_last_cuda_error(void) { return g_cuda_err; }

int spec_debug_build(void) {
#ifdef SPEC_DEBUG
    return 1;
#else
    return 0;
#endif
}

int spec_debug_failures(int* line) {
    using Reader = cudaError_t (*)(unsigned int*, unsigned int*);
    const Reader readers[] = {sv::debug_read_rows, sv::debug_read_rows_smem, sv::debug_read_argmax,
                              sv::debug_read_mentor, sv::debug_read_beta, sv::debug_read_tree_build};
    long long total = 0;
    int first = 0;
    for (const Reader rd : readers) {
        unsigned int c = 0u, l = 0u;
        if (rd(&c, &l) != cudaSuccess) return -1;
        if (c && !first) first = (int)l;
        total += c;
    }
    if (line) *line = first;
    return total > 0x7FFFFFFF ? 0x7FFFFFFF : (int)total;
}

size_t spec_verify_workspace_size(int B, int gamma, int V, spec_dtype dtype) {
    if (B < 1 || gamma < 1 || V < 1) return 0;
    return verify_ws(B, gamma, V, dtype).total;
}

spec_status spec_verify(const void* target, const void* draft, spec_dtype dtype,
                        const int32_t* draft_tokens, int B, int gamma, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset,
                        int32_t* accepted, int32_t* tokens, int32_t* next_token,
                        int32_t* status, float* probs_dbg,
                        void* workspace, size_t ws_bytes, spec_stream stream) {
    return verify_impl(target, draft, dtype, draft_tokens, B, gamma, V, sampling, seed, offset, accepted,
                       tokens, next_token, status, probs_dbg, workspace, ws_bytes, stream, 1.f);
}

spec_status spec_verify_lenient(const void* target, const void* draft, spec_dtype dtype,
                                const int32_t* draft_tokens, int B, int gamma, int V,
                                spec_sampling sampling, float lenience, uint64_t seed, uint64_t offset,
                                int32_t* accepted, int32_t* tokens, int32_t* next_token,
                                int32_t* status, float* probs_dbg,
                                void* workspace, size_t ws_bytes, spec_stream stream) {
    return verify_impl(target, draft, dtype, draft_tokens, B, gamma, V, sampling, seed, offset, accepted,
                       tokens, next_token, status, probs_dbg, workspace, ws_bytes, stream, lenience);
}

size_t spec_verify_tree_workspace_size(int B, int N, int V, spec_dtype dtype) {
    (void)dtype;
    if (B < 1 || N < 1 || V < 1) return 0;
    return ws_layout(B, N, V).total;
}

spec_status spec_verify_tree(const void* target, spec_dtype dtype, const int32_t* node_tokens,
                             const int32_t* parent, const int32_t* depth, int B, int N, int V,
                             int max_depth, int32_t* accept_len, int32_t* path_nodes,
                             int32_t* tokens, int32_t* bonus, int32_t* status,
                             void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype)) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || N < 1 || N > SPEC_MAX_TREE_N || V < 1 || V > SPEC_MAX_V ||
        max_depth < 0 || max_depth >= N)
        return SPEC_EINVAL;
    if (!target || !node_tokens || !parent || !depth || !accept_len || !path_nodes || !tokens ||
        !bonus || !workspace)
        return SPEC_EINVAL;
    if (!aligned(target, esize(dtype)) || !aligned(workspace, kAlign)) return SPEC_EINVAL;
    const Ws w = ws_layout(B, N, V);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    sv::ArgmaxParams p = {};
    p.logits = target;
    p.B = B;
    p.rows_per_b = N;
    p.V = V;
    p.mode = sv::kArgTree;
    p.max_depth = max_depth;
    p.node_tokens = node_tokens;
    p.parent = parent;
    p.depth = depth;
    p.out0 = accept_len;
    p.out1 = path_nodes;
    p.out2 = tokens;
    p.out3 = bonus;
    p.status = status;
    return launch_argmax_checked(p, dtype == SPEC_F32 ? 0 : 1, workspace, w,
                                 reinterpret_cast<cudaStream_t>(stream));
}

spec_status spec_tree_build(const int32_t* candidates, const int32_t* counts, const int32_t* root_token,
                            int B, int C, int L, int V, int N, int32_t* node_tokens, int32_t* parent,
                            int32_t* depth, uint8_t* mask, int32_t* n_nodes, int32_t* status,
                            spec_stream stream) {
    if (B < 1 || B > (1 << 24) || C < 1 || C > SPEC_MAX_TREE_C || L < 1 || L > SPEC_MAX_TREE_L ||
        C * L > SPEC_MAX_TREE_CL || V < 1 || N < 2 || N > SPEC_MAX_TREE_N)
        return SPEC_EINVAL;
    if (!candidates || !root_token || !node_tokens || !parent || !depth || !n_nodes) return SPEC_EINVAL;
    if (!aligned(candidates, 4) || !aligned(counts, 4) || !aligned(root_token, 4) || !aligned(node_tokens, 4) ||
        !aligned(parent, 4) || !aligned(depth, 4) || !aligned(n_nodes, 4) || !aligned(status, 4))
        return SPEC_EINVAL;
    const cudaError_t e = sv::launch_tree_build(candidates, counts, root_token, B, C, L, V, N, node_tokens, parent,
                                                depth, mask, n_nodes, status,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

spec_status spec_acceptance_rate(const void* target, const void* draft, spec_dtype dtype, int B, int gamma,
                                 int V, spec_sampling sampling, float* beta, int32_t* status,
                                 void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype) || !sampling_ok(sampling) || sampling.temperature <= 0.f) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V)
        return SPEC_EINVAL;
    if (!target || !draft || !beta || !workspace) return SPEC_EINVAL;
    const int es = esize(dtype);
    if (!aligned(target, es) || !aligned(draft, es) || !aligned(beta, 4) || !aligned(status, 4) ||
        !aligned(workspace, kAlign))
        return SPEC_EINVAL;
    const Ws w = ws_layout(B, 2 * gamma + 1, V);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    const float c2 = kLog2e / sampling.temperature;
    if (!std::isfinite(c2)) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int dt = dtype == SPEC_F32 ? 0 : 1;
    sv::RowParams p = {};
    p.target = target;
    p.draft = draft;
    p.draft_tokens = nullptr;  // records only: no acceptance test
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.rows_per_b = 2 * gamma + 1;
    p.mode = sv::kModeMentor;  // the row kernel writes the records and nothing else
    p.lenience = 1.f;
    p.transform = transform_bits(sampling, V);
    p.top_k = sampling.top_k;
    p.top_p = sampling.top_p;
    p.c2 = c2;
    p.status = status;
    spec_status s = run_rows(p, dt, workspace, w, st);
    if (s != SPEC_OK) return s;
    const cudaError_t e = sv::launch_beta(p, dt, beta, device_sms(), st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

size_t spec_verify_mentor_workspace_size(int B, int gamma, int V, spec_dtype dtype) {
    (void)dtype;
    if (B < 1 || gamma < 1 || V < 1) return 0;
    return mentor_ws(B, gamma, V).total;
}

spec_status spec_verify_mentor(const void* target, const void* draft, spec_dtype dtype,
                               const int32_t* draft_tokens, int B, int gamma, int V,
                               float temperature, float kl_bound, int bisect_iters,
                               uint64_t seed, uint64_t offset,
                               int32_t* accepted, int32_t* tokens, int32_t* next_token,
                               int32_t* status, float* alpha_out, float* beta_out,
                               float* probs_dbg,
                               void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype)) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V)
        return SPEC_EINVAL;
    if (!finite(temperature) || temperature <= 0.f || !finite(kl_bound) || kl_bound < 0.f ||
        bisect_iters < 1 || bisect_iters > SPEC_MAX_BISECT)
        return SPEC_EINVAL;
    if (!target || !draft || !draft_tokens || !accepted || !tokens || !next_token || !workspace)
        return SPEC_EINVAL;
    const int es = esize(dtype);
    if (!aligned(target, es) || !aligned(draft, es) || !aligned(workspace, kAlign)) return SPEC_EINVAL;
    const MentorWs w = mentor_ws(B, gamma, V);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    const float c2 = kLog2e / temperature;
    if (!std::isfinite(c2)) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int dt = dtype == SPEC_F32 ? 0 : 1;

    sv::RowParams p = {};
    p.target = target;
    p.draft = draft;
    p.draft_tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.rows_per_b = 2 * gamma + 1;
    p.mode = sv::kModeMentor;
    p.lenience = 1.f;
    p.transform = 0;
    p.top_p = 1.f;
    p.c2 = c2;
    p.seed = seed;
    p.offset = offset;
    spec_status s = run_rows(p, dt, workspace, w.lin, st);
    if (s != SPEC_OK) return s;

    sv::MentorParams m = {};
    m.target = target;
    m.draft = draft;
    m.B = B;
    m.gamma = gamma;
    m.V = V;
    m.bf16 = dtype == SPEC_BF16;
    m.c2 = c2;
    m.inv_t = 1.f / temperature;
    m.kl_bound = kl_bound;
    m.iters = bisect_iters;
    m.seed = seed;
    m.offset = offset;
    m.rows = at<sv::RowRec>(workspace, w.lin.rows);
    m.keys = at<uint32_t>(workspace, w.keys);
    m.idx = at<uint32_t>(workspace, w.idx);
    m.arr = at<float>(workspace, w.arr);
    // both cleared with the row kernel's control; mentor mode uses neither
    m.work = at<unsigned int>(workspace, w.lin.work) + 1;
    m.rejmark = at<unsigned int>(workspace, w.lin.seq_cnt);
    m.pos_state = at<int32_t>(workspace, w.pos_state);
    m.pos_beta = at<float>(workspace, w.pos_beta);
    m.pos_scale = at<float>(workspace, w.pos_scale);
    m.accepted = accepted;
    m.tokens = tokens;
    m.next_token = next_token;
    m.status = status;
    m.alpha_out = alpha_out;
    m.beta_out = beta_out;
    m.probs_dbg = probs_dbg;
    const cudaError_t e = sv::launch_mentor(m, std::min(w.slots, device_sms()), device_sms() * 8, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

size_t spec_sample_workspace_size(int B, int P, int V, spec_dtype dtype) {
    (void)dtype;
    if (B < 1 || P < 1 || V < 1) return 0;
    return ws_layout(B, P, V).total;
}

spec_status spec_sample(const void* logits, spec_dtype dtype, int B, int P, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset, uint32_t pos0,
                        uint32_t purpose, int32_t* tokens_out, int32_t* status,
                        void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype) || !sampling_ok(sampling)) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || P < 1 || P > 1024 || V < 1 || V > SPEC_MAX_V) return SPEC_EINVAL;
    if (!logits || !tokens_out || !workspace) return SPEC_EINVAL;
    if (!aligned(logits, esize(dtype)) || !aligned(workspace, kAlign)) return SPEC_EINVAL;
    const Ws w = ws_layout(B, P, V);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int dt = dtype == SPEC_F32 ? 0 : 1;
    if (sampling.temperature == 0.f) {
        sv::ArgmaxParams p = {};
        p.logits = logits;
        p.B = B;
        p.rows_per_b = P;
        p.V = V;
        p.mode = sv::kArgSample;
        p.out0 = tokens_out;
        p.status = status;
        return launch_argmax_checked(p, dt, workspace, w, st);
    }
    if (status) {
        const cudaError_t e = cudaMemsetAsync(status, 0, (size_t)B * sizeof(int32_t), st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    sv::RowParams p = {};
    p.target = logits;
    p.B = B;
    p.gamma = 0;
    p.V = V;
    p.rows_per_b = P;
    p.mode = sv::kModeSample;
    p.lenience = 1.f;
    p.transform = transform_bits(sampling, V);
    p.top_k = sampling.top_k;
    p.top_p = sampling.top_p;
    p.c2 = kLog2e / sampling.temperature;
    if (!std::isfinite(p.c2)) return SPEC_EINVAL;
    p.seed = seed;
    p.offset = offset;
    p.pos0 = pos0;
    p.purpose = purpose;
    p.status = status;
    p.sample_out = tokens_out;
    return run_rows(p, dt, workspace, w, st);
}

spec_status spec_philox_uniform(uint64_t seed, uint64_t row0, uint32_t position, uint32_t purpose,
                                int n, float* out, spec_stream stream) {
    if (n < 1 || n > (1 << 30) || !out || !aligned(out, 4)) return SPEC_EINVAL;
    philox_uniform_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        seed, row0, position, purpose, n, out);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

}  // extern "C"
