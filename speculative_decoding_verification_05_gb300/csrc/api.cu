// C ABI of libspecverify: argument validation, workspace layout, launch
// configuration. Every entry point checks its arguments on the host before
// touching CUDA, so invalid calls return SPEC_EINVAL with nothing enqueued.

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "specverify.h"

namespace sv {
size_t mentor_smem_bytes(int V);
spec_status note_cuda_error(cudaError_t e);
}

namespace {

thread_local char g_cuda_err[256] = "";

constexpr size_t kAlign = 256;
constexpr int kMentorSlots = 128;

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

// Every layout starts with the control region that must be zero when the
// kernels start (arrival counters, packed per-row argmaxes); each call clears
// it with one memset, so the workspace may hold anything on entry. Records and
// scratch follow and are always written before they are read.
struct LinearWs {
    size_t cnt, cnt64, rowbest, rowbad, zero_end, recs, total;
};

LinearWs linear_ws(int B, int rows_per_b) {
    LinearWs w;
    size_t o = 0;
    const size_t rows = (size_t)B * rows_per_b;
    w.cnt = o;
    o = al(o + (size_t)B * sizeof(unsigned int));
    w.cnt64 = o;
    o = al(o + (size_t)B * sizeof(unsigned long long));
    w.rowbest = o;
    o = al(o + rows * sizeof(unsigned long long));
    w.rowbad = o;
    o = al(o + rows * sizeof(unsigned int));
    w.zero_end = o;
    w.recs = o;
    o = al(o + rows * sizeof(sv::TaskRec));
    w.total = o;
    return w;
}

spec_status clear_control(void* ws, const LinearWs& w, cudaStream_t st) {
    const cudaError_t e = cudaMemsetAsync(ws, 0, w.zero_end, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

struct MentorWs {
    LinearWs lin;
    size_t mflags, mtok, mcnt, keys, idx, arr, total;
    int slots;
};

MentorWs mentor_ws(int B, int gamma, int V) {
    MentorWs w;
    w.lin = linear_ws(B, gamma + 1);
    size_t o = w.lin.total;
    const size_t t = (size_t)B * gamma;
    w.slots = (int)std::min<size_t>(t, kMentorSlots);
    w.mcnt = w.lin.cnt;  // the row kernel leaves cnt alone in mentor mode
    w.mflags = o;
    o = al(o + t * 4);
    w.mtok = o;
    o = al(o + t * 4);
    w.keys = o;
    o = al(o + (size_t)w.slots * 2 * V * 4);
    w.idx = o;
    o = al(o + (size_t)w.slots * 2 * V * 4);
    w.arr = o;
    o = al(o + (size_t)w.slots * 7 * V * 4);
    w.total = o;
    return w;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

// ---- launch configuration ---------------------------------------------------

// Cluster size C and slice length L for the row kernel: the smallest C whose
// per-CTA shared memory stays within 72 KB (three CTAs per SM), else the
// smallest C within 200 KB; 0 if V is too large.
int pick_cluster(int dtype, int V, bool two_rows, int* L, size_t* smem) {
    for (int pass = 0; pass < 2; ++pass) {
        const size_t cap = pass == 0 ? 72 * 1024 : 200 * 1024;
        for (int C = 1; C <= 16; C *= 2) {
            const int l = (((V + C - 1) / C) + 15) & ~15;
            if ((long long)l * (C - 1) >= V && C > 1) break;  // last CTA would be empty
            const size_t sm = sv::rows_smem_bytes(dtype, l, two_rows);
            if (sm <= cap) {
                *L = l;
                *smem = sm;
                return C;
            }
        }
    }
    return 0;
}

spec_status launch_rows_checked(sv::RowParams& p, int dtype, int num_tasks, bool two_rows,
                                cudaStream_t st) {
    int L;
    size_t smem;
    const int C = pick_cluster(dtype, p.V, two_rows, &L, &smem);
    if (!C) return SPEC_EINVAL;
    if ((long long)num_tasks * C > 0x7FFFFFFFLL) return SPEC_EINVAL;
    p.C = C;
    p.L = L;
    const cudaError_t e = sv::launch_rows(p, dtype, num_tasks, smem, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

spec_status launch_argmax_checked(sv::ArgmaxParams& p, int dtype, cudaStream_t st) {
    const long long total = (long long)p.B * p.rows_per_b * p.V;
    long long grid = std::min<long long>((long long)device_sms() * 4, (total + 8191) / 8192);
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
    }
    return "SPEC_UNKNOWN";
}

const char* spec_last_cuda_error(void) { return g_cuda_err; }

size_t spec_verify_workspace_size(int B, int gamma, int V, spec_dtype dtype) {
    (void)V;
    (void)dtype;
    if (B < 1 || gamma < 1) return 0;
    return linear_ws(B, gamma + 1).total;
}

spec_status spec_verify(const void* target, const void* draft, spec_dtype dtype,
                        const int32_t* draft_tokens, int B, int gamma, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset,
                        int32_t* accepted, int32_t* tokens, int32_t* next_token,
                        int32_t* status, float* probs_dbg,
                        void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype) || !sampling_ok(sampling)) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V)
        return SPEC_EINVAL;
    const bool greedy = sampling.temperature == 0.f;
    if (!target || (!greedy && !draft) || !draft_tokens || !accepted || !tokens || !next_token || !workspace)
        return SPEC_EINVAL;
    const int es = esize(dtype);
    if (!aligned(target, es) || (draft && !aligned(draft, es)) || !aligned(workspace, kAlign))
        return SPEC_EINVAL;
    const LinearWs w = linear_ws(B, gamma + 1);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (spec_status c = clear_control(workspace, w, st)) return c;

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
        p.rowbest = at<unsigned long long>(workspace, w.rowbest);
        p.rowbad = at<unsigned int>(workspace, w.rowbad);
        p.cnt = at<unsigned long long>(workspace, w.cnt64);
        return launch_argmax_checked(p, dtype == SPEC_F32 ? 0 : 1, st);
    }
    sv::RowParams p = {};
    p.target = target;
    p.draft = draft;
    p.draft_tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.rows_per_b = gamma + 1;
    p.mode = sv::kModeVerify;
    p.transform = transform_bits(sampling, V);
    p.top_k = sampling.top_k;
    p.top_p = sampling.top_p;
    p.c2 = kLog2e / sampling.temperature;
    p.seed = seed;
    p.offset = offset;
    p.wait_limit = 1u << 26;
    p.accepted = accepted;
    p.tokens = tokens;
    p.next_token = next_token;
    p.status = status;
    p.probs_dbg = probs_dbg;
    p.recs = at<sv::TaskRec>(workspace, w.recs);
    p.cnt = at<unsigned int>(workspace, w.cnt);
    if (!std::isfinite(p.c2)) return SPEC_EINVAL;
    return launch_rows_checked(p, dtype == SPEC_F32 ? 0 : 1, B * (gamma + 1), true, st);
}

size_t spec_verify_tree_workspace_size(int B, int N, int V, spec_dtype dtype) {
    (void)V;
    (void)dtype;
    if (B < 1 || N < 1) return 0;
    return linear_ws(B, N).total;
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
    const LinearWs w = linear_ws(B, N);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    if (spec_status c = clear_control(workspace, w, reinterpret_cast<cudaStream_t>(stream))) return c;
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
    p.rowbest = at<unsigned long long>(workspace, w.rowbest);
    p.rowbad = at<unsigned int>(workspace, w.rowbad);
    p.cnt = at<unsigned long long>(workspace, w.cnt64);
    return launch_argmax_checked(p, dtype == SPEC_F32 ? 0 : 1, reinterpret_cast<cudaStream_t>(stream));
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
    if (spec_status c = clear_control(workspace, w.lin, st)) return c;

    sv::RowParams p = {};
    p.target = target;
    p.draft = draft;
    p.draft_tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.rows_per_b = gamma + 1;
    p.mode = sv::kModeMentor;
    p.transform = 0;
    p.top_p = 1.f;
    p.c2 = c2;
    p.seed = seed;
    p.offset = offset;
    p.wait_limit = 1u << 26;
    p.probs_dbg = probs_dbg;
    p.recs = at<sv::TaskRec>(workspace, w.lin.recs);
    p.cnt = at<unsigned int>(workspace, w.lin.cnt);
    spec_status s = launch_rows_checked(p, dtype == SPEC_F32 ? 0 : 1, B * (gamma + 1), true, st);
    if (s != SPEC_OK) return s;

    sv::MentorParams m = {};
    m.target = target;
    m.draft = draft;
    m.draft_tokens = draft_tokens;
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
    m.recs = at<sv::TaskRec>(workspace, w.lin.recs);
    m.m_flags = at<int32_t>(workspace, w.mflags);
    m.m_token = at<int32_t>(workspace, w.mtok);
    m.cnt = at<unsigned int>(workspace, w.mcnt);
    m.keys = at<uint32_t>(workspace, w.keys);
    m.idx = at<uint32_t>(workspace, w.idx);
    m.arr = at<float>(workspace, w.arr);
    m.accepted = accepted;
    m.tokens = tokens;
    m.next_token = next_token;
    m.status = status;
    m.alpha_out = alpha_out;
    m.beta_out = beta_out;
    m.probs_dbg = probs_dbg;
    const cudaError_t e = sv::launch_mentor(m, w.slots, st);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

size_t spec_sample_workspace_size(int B, int P, int V, spec_dtype dtype) {
    (void)V;
    (void)dtype;
    if (B < 1 || P < 1) return 0;
    return linear_ws(B, P).total;
}

spec_status spec_sample(const void* logits, spec_dtype dtype, int B, int P, int V,
                        spec_sampling sampling, uint64_t seed, uint64_t offset, uint32_t pos0,
                        uint32_t purpose, int32_t* tokens_out, int32_t* status,
                        void* workspace, size_t ws_bytes, spec_stream stream) {
    if (!dtype_ok(dtype) || !sampling_ok(sampling)) return SPEC_EINVAL;
    if (B < 1 || B > (1 << 24) || P < 1 || P > 1024 || V < 1 || V > SPEC_MAX_V) return SPEC_EINVAL;
    if (!logits || !tokens_out || !workspace) return SPEC_EINVAL;
    if (!aligned(logits, esize(dtype)) || !aligned(workspace, kAlign)) return SPEC_EINVAL;
    const LinearWs w = linear_ws(B, P);
    if (ws_bytes < w.total) return SPEC_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (spec_status c = clear_control(workspace, w, st)) return c;
    if (sampling.temperature == 0.f) {
        sv::ArgmaxParams p = {};
        p.logits = logits;
        p.B = B;
        p.rows_per_b = P;
        p.V = V;
        p.mode = sv::kArgSample;
        p.out0 = tokens_out;
        p.status = status;
        p.rowbest = at<unsigned long long>(workspace, w.rowbest);
        p.rowbad = at<unsigned int>(workspace, w.rowbad);
        p.cnt = at<unsigned long long>(workspace, w.cnt64);
        return launch_argmax_checked(p, dtype == SPEC_F32 ? 0 : 1, st);
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
    p.transform = transform_bits(sampling, V);
    p.top_k = sampling.top_k;
    p.top_p = sampling.top_p;
    p.c2 = kLog2e / sampling.temperature;
    if (!std::isfinite(p.c2)) return SPEC_EINVAL;
    p.seed = seed;
    p.offset = offset;
    p.pos0 = pos0;
    p.purpose = purpose;
    p.wait_limit = 1u << 26;
    p.status = status;
    p.sample_out = tokens_out;
    return launch_rows_checked(p, dtype == SPEC_F32 ? 0 : 1, B * P, false, st);
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
