// store_kvcache: the slot scatter of new K/V rows into the paged cache
// ("3.3 Model skeleton and core operators", sec. 7.1; "Nano-vLLM 源码解读
// 第17篇", sec. 5.1).  One warp per token moves the token's D-element key and
// value rows as 16-byte vectors: all loads of the warp are issued before its
// stores, so each warp keeps 2 * D * 2 bytes in flight.  It is a bit copy.
#include "common.cuh"
#include "internal.h"

namespace nvattn {

constexpr int kStoreThreads = 256;
constexpr int kStoreMaxVecPerLane = 8;   // D <= 2048 handled in one pass

__global__ void __launch_bounds__(kStoreThreads)
store_kvcache_kernel(const uint4 *__restrict__ key, int64_t key_stride_v,
                     const uint4 *__restrict__ value, int64_t value_stride_v,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int32_t *__restrict__ slot_mapping, int64_t N, int vec_per_row,
                     int64_t num_slots, int *err_count) {
    pdl_wait_release();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kStoreThreads / 32);
    for (int64_t n = ((int64_t)blockIdx.x * kStoreThreads + threadIdx.x) >> 5; n < N;
         n += warps) {
        const int64_t slot = __ldg(slot_mapping + n);
        if (slot == -1) continue;                       // padding token
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0) count_error(err_count);
            continue;
        }
        for (int base = 0; base < vec_per_row; base += 32 * kStoreMaxVecPerLane) {
            uint4 kv[kStoreMaxVecPerLane], vv[kStoreMaxVecPerLane];
#pragma unroll
            for (int u = 0; u < kStoreMaxVecPerLane; ++u) {
                const int c = base + lane + 32 * u;
                if (c < vec_per_row) {
                    kv[u] = __ldg(key + n * key_stride_v + c);
                    vv[u] = __ldg(value + n * value_stride_v + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kStoreMaxVecPerLane; ++u) {
                const int c = base + lane + 32 * u;
                if (c < vec_per_row) {
                    k_cache[slot * vec_per_row + c] = kv[u];
                    v_cache[slot * vec_per_row + c] = vv[u];
                }
            }
        }
    }
}

cudaError_t launch_store_kvcache(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                                 int64_t value_stride, uint16_t *k_cache, uint16_t *v_cache,
                                 const int32_t *slot_mapping, int64_t N, int D,
                                 int64_t num_slots, int *err_count, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int warps_per_block = kStoreThreads / 32;
    int64_t blocks = (N + warps_per_block - 1) / warps_per_block;
    if (blocks > 152 * 32) blocks = 152 * 32;
    return launch_pdl(store_kvcache_kernel, dim3((unsigned)blocks), dim3(kStoreThreads), (size_t)0,
                      s, (const uint4 *)key, key_stride / 8, (const uint4 *)value,
                      value_stride / 8, (uint4 *)k_cache, (uint4 *)v_cache, slot_mapping, N,
                      D / 8, num_slots, err_count);
}

}  // namespace nvattn
