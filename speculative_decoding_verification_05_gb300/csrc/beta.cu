// Per-position acceptance probability of speculative sampling.
//
// "Fast Inference from Transformers via Speculative Decoding", section
// "方法细节" (接受率精确刻画): a draft token drawn from p is accepted with
// probability beta = sum_x min(q(x), p(x)), and the acceptance rate alpha is
// its expectation over positions ("Accelerating Large Language Model Decoding
// with Speculative Sampling", appendix proof of Theorem 1, gives the same sum
// as one minus the rejection probability).
//
// The row kernel (records only) has written every row's maximum, sum,
// threshold and kept mass; this kernel streams each (target k, draft k) row
// pair once more and sums min(q, p) over the transformed distributions, each
// thread over its elements left to right, then a butterfly in each warp, then
// the warps in order, so the result does not depend on timing.

#include <algorithm>

#include "common.cuh"
#include "draw.cuh"

namespace sv {
namespace {

constexpr int BT = kDrawNT;

template <typename E>
__global__ void __launch_bounds__(BT) beta_kernel(const __grid_constant__ RowParams p, float* beta) {
    __shared__ float red[BT / 32];
    __shared__ int job;
    constexpr int PER = draw_per<E>();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.gamma, G1 = G + 1, R = p.rows_per_b, V = p.V;
    const long long jobs = (long long)p.B * G;
    const E* tgt = reinterpret_cast<const E*>(p.target);
    const E* dft = reinterpret_cast<const E*>(p.draft);
    unsigned* counter = p.work + 1;
    for (;;) {
        if (tid == 0) job = (int)atomicAdd(counter, 1u);
        __syncthreads();
        const long long jb = job;
        if (jb >= jobs) break;
        const int b = (int)(jb / G), k = (int)(jb - (long long)b * G);
        const RowRec* rb = p.rows + (size_t)b * R;
        const RowRec t = load_rec(rb + k), d = load_rec(rb + G1 + k);
        const bool bad = ((t.flags | d.flags) & kRecEData) != 0;
        const KeptExp qf{t.thr, p.c2, t.m * p.c2, 1.f / t.Sk}, pf{d.thr, p.c2, d.m * p.c2, 1.f / d.Sk};
        const E* rt = tgt + ((size_t)b * G1 + k) * V;
        const E* rd = dft + ((size_t)b * G + k) * V;
        float acc = 0.f;
        constexpr int VE = 16 / (int)sizeof(E);
        constexpr int U = 4;  // 16-byte vectors of each row in flight per thread
        const bool vec = (((uintptr_t)rt | (uintptr_t)rd) & 15) == 0;
        if (!bad && vec) {
            // both rows start on 16 bytes: raw vectors, U of each in flight
            const int nb = V / VE;
            const uint4* vt = reinterpret_cast<const uint4*>(rt);
            const uint4* vd = reinterpret_cast<const uint4*>(rd);
            for (int j = tid; j < nb; j += BT * U) {
                uint4 a[U], c[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (j + u * BT < nb) {
                        a[u] = ld_stream_v4(vt + j + u * BT);
                        c[u] = ld_stream_v4(vd + j + u * BT);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (j + u * BT < nb) {
                        float xt[VE], xd[VE];
                        VecTraits<E>::unpack(a[u], xt);
                        VecTraits<E>::unpack(c[u], xd);
#pragma unroll
                        for (int e = 0; e < VE; ++e) acc += fminf(qf(xt[e]), pf(xd[e]));
                    }
                }
            }
            for (int i = nb * VE + tid; i < V; i += BT)
                acc += fminf(qf(VecTraits<E>::load1(rt + i)), pf(VecTraits<E>::load1(rd + i)));
        } else if (!bad) {
            for (int i0 = tid * PER; i0 < V; i0 += BT * PER) {
                float xt[PER], xd[PER];
                draw_load<E>(rt, i0, V, xt);
                draw_load<E>(rd, i0, V, xd);
#pragma unroll
                for (int e = 0; e < PER; ++e) acc += i0 + e < V ? fminf(qf(xt[e]), pf(xd[e])) : 0.f;
            }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < BT / 32; ++w) s += red[w];
            if (SV_IN(jb, (long long)p.B * p.gamma)) beta[jb] = bad ? NAN : s;
            if (k == 0 && p.status) {
                int fl = 0;
                for (int i = 0; i < R; ++i) fl |= __ldcg(&rb[i].flags);
                p.status[b] = (fl & kRecEData) ? kEData : kOk;
            }
        }
        __syncthreads();
    }
}

template <typename E>
cudaError_t launch_beta_t(const RowParams& p, float* beta, int sms, cudaStream_t stream) {
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, beta_kernel<E>, BT, 0) != cudaSuccess || n < 1) n = 1;
        return n;
    }();
    const long long jobs = (long long)p.B * p.gamma;
    const int grid = (int)std::min<long long>(jobs, (long long)sms * per_sm);
    beta_kernel<E><<<grid, BT, 0, stream>>>(p, beta);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_beta(const RowParams& p, int dtype, float* beta, int sms, cudaStream_t stream) {
    return dtype == 0 ? launch_beta_t<float>(p, beta, sms, stream) : launch_beta_t<bf16_t>(p, beta, sms, stream);
}

SV_DEBUG_READER(beta)

}  // namespace sv
