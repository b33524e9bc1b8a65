// spec_verify_noalloc: spec_verify for callers that cannot allocate device
// memory.
//
// Some callers of a verification step are not allowed to call cudaMalloc or
// any allocating routine at the point where they verify: an inference engine
// plugin whose host framework owns every device allocation and forbids
// allocation inside its execute callback, a server that fixes its device
// memory budget at start-up and must never allocate on the request path, or a
// C program that links this library without a device allocator of its own.
// For them this entry point takes no workspace: its scratch memory is one
// file-scope __device__ array of a fixed size, which every GPU that loads the
// library holds until the process exits. Everything else is spec_verify's
// path, unchanged: the same kernels, the same outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents; spec_verify clears the part that must start at zero (its control
// region) at the start of each call. Calls that overlap on the GPU (on
// different streams, or from different host threads without ordering) race
// on the array and must be avoided.

#include <mutex>

#include "common.cuh"
#include "specverify.h"

namespace sv {
spec_status note_cuda_error(cudaError_t e);
}

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device with that device current. In host code the array's name is only
// a host-side stand-in; the kernels must be given this address. Under lazy
// module loading the lookup is also what loads this file's module and commits
// the array's memory, so the first call belongs at start-up. The address is
// cached for the life of the process: a device reset after the first call
// would leave it stale, and is not supported.
spec_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return sv::note_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return SPEC_EINVAL;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return sv::note_cuda_error(e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_verify_noalloc(const void* target, const void* draft, spec_dtype dtype,
                                           const int32_t* draft_tokens, int B, int gamma, int V,
                                           spec_sampling sampling, uint64_t seed, uint64_t offset,
                                           int32_t* accepted, int32_t* tokens, int32_t* next_token,
                                           int32_t* status, float* probs_dbg, spec_stream stream) {
    const size_t need = spec_verify_workspace_size(B, gamma, V, dtype);
    if (need == 0 || need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_EINVAL;
    void* ws = nullptr;
    if (spec_status s = scratch_address(&ws)) return s;
    return spec_verify(target, draft, dtype, draft_tokens, B, gamma, V, sampling, seed, offset,
                       accepted, tokens, next_token, status, probs_dbg, ws,
                       (size_t)SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
