// SiluAndMul, the SwiGLU activation of the Qwen3 MLP ("3.3 Model skeleton
// and core operators", sec. 4 and 5): row t of the merged gate_up output holds
// the gate in its first I elements and the up projection in its last I, and
// out[t][i] = silu(gate_i) * up_i, computed in fp32 and rounded once to bf16.
// Pure streaming: every input byte is read once and every output byte written
// once, so the kernel is HBM-bound.  A thread moves 16-byte vectors (eight
// elements of gate and the matching eight of up), walking them with the
// grid's stride, and loads its next kSwigluPipe vectors before it computes
// and stores the current ones, so loads stay in flight while it computes; the
// grid is one resident wave (four 256-thread blocks per SM at 64 registers).
#include "common.cuh"
#include "internal.h"

namespace nvattn {

constexpr int kSwigluThreads = 256;
constexpr int kSwigluPipe = 2;

__device__ __forceinline__ float silu_times(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

// (token, vector) of a flat vector index, advanced by a fixed stride without
// a 64-bit division per step.
struct VecCursor {
    int64_t t;
    int c;
    __device__ __forceinline__ void advance(int64_t dt, int dc, int nvec) {
        t += dt;
        c += dc;
        if (c >= nvec) {
            c -= nvec;
            ++t;
        }
    }
};

// `out` may be `x` itself (same token stride): element (t, i) of the output
// then overwrites gate (t, i), which only the same thread has read.
__global__ void __launch_bounds__(kSwigluThreads)
silu_and_mul_kernel(const uint4 *x, int64_t x_stride_v, uint4 *out, int64_t out_stride_v,
                    int64_t T, int nvec) {
    pdl_wait_release();
    const int64_t total = T * nvec;
    const int64_t stride = (int64_t)gridDim.x * kSwigluThreads;
    const int64_t dt = stride / nvec;
    const int dc = (int)(stride - dt * nvec);
    int64_t idx = (int64_t)blockIdx.x * kSwigluThreads + threadIdx.x;
    if (idx >= total) return;
    VecCursor cur{idx / nvec, (int)(idx % nvec)};
    VecCursor ahead = cur;
    uint4 g[kSwigluPipe], u[kSwigluPipe];
    // The next kSwigluPipe vectors of this thread are loaded before the current
    // ones are computed and stored.
#pragma unroll
    for (int k = 0; k < kSwigluPipe; ++k) {
        if (idx + k * stride < total) {
            const uint4 *row = x + ahead.t * x_stride_v;
            g[k] = row[ahead.c];
            u[k] = row[nvec + ahead.c];
        }
        ahead.advance(dt, dc, nvec);
    }
    for (; idx < total; idx += kSwigluPipe * stride) {
        uint4 ng[kSwigluPipe], nu[kSwigluPipe];
#pragma unroll
        for (int k = 0; k < kSwigluPipe; ++k) {
            if (idx + (kSwigluPipe + k) * stride < total) {
                const uint4 *row = x + ahead.t * x_stride_v;
                ng[k] = row[ahead.c];
                nu[k] = row[nvec + ahead.c];
            }
            ahead.advance(dt, dc, nvec);
        }
#pragma unroll
        for (int k = 0; k < kSwigluPipe; ++k) {
            if (idx + k * stride < total) {
                const uint32_t gw[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
                const uint32_t uw[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = pack_bf16x2(silu_times(bf16_lo(gw[e]), bf16_lo(uw[e])),
                                       silu_times(bf16_hi(gw[e]), bf16_hi(uw[e])));
                out[cur.t * out_stride_v + cur.c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            cur.advance(dt, dc, nvec);
            g[k] = ng[k];
            u[k] = nu[k];
        }
    }
}

cudaError_t launch_silu_and_mul(const uint16_t *x, int64_t x_stride, uint16_t *out,
                                int64_t out_stride, int64_t T, int I, cudaStream_t s) {
    const int nvec = I / 8;
    const int64_t total = T * nvec;
    if (total == 0) return cudaSuccess;
    const int64_t per_block = (int64_t)kSwigluThreads * kSwigluPipe;
    int64_t blocks = (total + per_block - 1) / per_block;
    static const int64_t wave = resident_grid(silu_and_mul_kernel, kSwigluThreads, 4);
    if (blocks > wave) blocks = wave;
    return launch_pdl(silu_and_mul_kernel, dim3((unsigned)blocks), dim3(kSwigluThreads), (size_t)0,
                      s, (const uint4 *)x, x_stride / 8, (uint4 *)out, out_stride / 8, T, nvec);
}

}  // namespace nvattn
