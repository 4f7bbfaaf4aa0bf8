// SiluAndMul, the SwiGLU activation of the Qwen3 MLP ("3.3 Model skeleton
// and core operators", sec. 4 and 5): row t of the merged gate_up output holds
// the gate in its first I elements and the up projection in its last I, and
// out[t][i] = silu(gate_i) * up_i, computed in fp32 and rounded once to bf16.
// Pure streaming: every input byte is read once and every output byte written
// once, so the kernel is HBM-bound.  A thread moves 16-byte vectors (eight
// elements of gate and the matching eight of up) and keeps kUnroll of them in
// flight; the grid is a whole number of waves over the 152 SMs.
#include "common.cuh"
#include "internal.h"

namespace nvattn {

constexpr int kSwigluThreads = 256;
constexpr int kSwigluUnroll = 4;
constexpr int kSwigluBlocksPerSm = 4;   // 64 registers x 256 threads: four resident
constexpr int kNumSms = 152;

__device__ __forceinline__ float silu_times(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

// `out` may be `x` itself (same token stride): element (t, i) of the output
// then overwrites gate (t, i), which only the same thread has read.
__global__ void __launch_bounds__(kSwigluThreads)
silu_and_mul_kernel(const uint4 *x, int64_t x_stride_v, uint4 *out, int64_t out_stride_v,
                    int64_t T, int nvec) {
    pdl_wait_release();
    const int64_t total = T * nvec;
    const int64_t stride = (int64_t)gridDim.x * kSwigluThreads;
    for (int64_t base = (int64_t)blockIdx.x * kSwigluThreads + threadIdx.x; base < total;
         base += stride * kSwigluUnroll) {
        uint4 g[kSwigluUnroll], u[kSwigluUnroll];
        int64_t t[kSwigluUnroll], c[kSwigluUnroll];
#pragma unroll
        for (int k = 0; k < kSwigluUnroll; ++k) {
            const int64_t idx = base + k * stride;
            t[k] = idx / nvec;
            c[k] = idx - t[k] * nvec;
            if (idx < total) {
                const uint4 *row = x + t[k] * x_stride_v;
                g[k] = row[c[k]];
                u[k] = row[nvec + c[k]];
            }
        }
#pragma unroll
        for (int k = 0; k < kSwigluUnroll; ++k) {
            if (base + k * stride < total) {
                const uint32_t gw[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
                const uint32_t uw[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = pack_bf16x2(silu_times(bf16_lo(gw[e]), bf16_lo(uw[e])),
                                       silu_times(bf16_hi(gw[e]), bf16_hi(uw[e])));
                out[t[k] * out_stride_v + c[k]] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

cudaError_t launch_silu_and_mul(const uint16_t *x, int64_t x_stride, uint16_t *out,
                                int64_t out_stride, int64_t T, int I, cudaStream_t s) {
    const int nvec = I / 8;
    const int64_t total = T * nvec;
    if (total == 0) return cudaSuccess;
    const int64_t per_block = (int64_t)kSwigluThreads * kSwigluUnroll;
    int64_t blocks = (total + per_block - 1) / per_block;
    const int64_t wave = (int64_t)kNumSms * kSwigluBlocksPerSm;
    if (blocks > wave) blocks = wave;
    return launch_pdl(silu_and_mul_kernel, dim3((unsigned)blocks), dim3(kSwigluThreads), (size_t)0,
                      s, (const uint4 *)x, x_stride / 8, (uint4 *)out, out_stride / 8, T, nvec);
}

}  // namespace nvattn
