// Host-side interface between the ABI translation unit (abi.cu, which checks
// arguments) and the translation units that own each kernel.  Launchers
// assume their arguments were already validated and return the
// cudaGetLastError() of their launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace nvattn {

// Blocks of `kernel` (with `threads` threads and no dynamic shared memory)
// resident at once on the current device: grid-stride kernels launch one
// such wave.  Falls back to 152 SMs x `fallback_per_sm` if a query fails.
template <typename... KArgs>
inline int64_t resident_grid(void (*kernel)(KArgs...), int threads, int fallback_per_sm) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) !=
            cudaSuccess || sms <= 0 || per_sm <= 0)
        return (int64_t)152 * fallback_per_sm;
    return (int64_t)sms * per_sm;
}

// Allows `kernel` `bytes` of dynamic shared memory on the current device.
// The attribute belongs to each device's context, so it is set once per
// device (bit d of `done` for device d < 64; always for higher ordinals);
// `force` sets it again (a launch found it missing: the device was reset).
template <typename... KArgs>
inline cudaError_t ensure_dynamic_smem(void (*kernel)(KArgs...), int bytes,
                                       std::atomic<uint64_t> &done, bool force = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (!force && bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

// Launch with programmatic stream serialization (see pdl_wait_release).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}


cudaError_t launch_rope_cos_sin(float *cos_sin, int max_position, int rotary_dim, double base,
                                cudaStream_t s);

cudaError_t launch_add_rmsnorm(const uint16_t *x, const uint16_t *residual,
                               const uint16_t *weight, uint16_t *out, uint16_t *residual_out,
                               int64_t T, int H, int64_t row_stride, float eps, cudaStream_t s);

cudaError_t launch_qknorm_rope(uint16_t *q, int64_t q_stride, uint16_t *k, int64_t k_stride,
                               const uint16_t *qw, const uint16_t *kw, const float *cos_sin,
                               int max_position, const int64_t *positions, int64_t T, int Hq,
                               int Hkv, float eps, int *err_count, cudaStream_t s);

cudaError_t launch_qknorm_rope_store(uint16_t *q, int64_t q_stride, uint16_t *k,
                                     int64_t k_stride, const uint16_t *v, int64_t v_stride,
                                     const uint16_t *qw, const uint16_t *kw,
                                     const float *cos_sin, int max_position,
                                     const int64_t *positions, const int32_t *slot_mapping,
                                     uint16_t *k_cache, uint16_t *v_cache, int64_t num_slots,
                                     int64_t T, int Hq, int Hkv, float eps, int write_k,
                                     int *err_count, cudaStream_t s);

// One bounded mbarrier wait that cannot succeed (about a second); records
// kPipelineFailureBit in err_count when it gives up.
cudaError_t launch_wait_timeout_selftest(int *err_count, cudaStream_t s);

cudaError_t launch_silu_and_mul(const uint16_t *x, int64_t x_stride, uint16_t *out,
                                int64_t out_stride, int64_t T, int I, cudaStream_t s);

cudaError_t launch_store_kvcache(const uint16_t *key, int64_t key_stride, const uint16_t *value,
                                 int64_t value_stride, uint16_t *k_cache, uint16_t *v_cache,
                                 const int32_t *slot_mapping, int64_t N, int D,
                                 int64_t num_slots, int *err_count, cudaStream_t s);

// ------------------------------------------------------------------ decode
struct DecodeParams {
    const uint16_t *q;
    int64_t q_stride;
    const int32_t *block_tables;
    int max_blocks;
    const int32_t *context_lens;
    uint16_t *o;
    int B, Hq, Hkv, block_size;
    int64_t num_blocks;
    float scale_log2;          // softmax_scale * log2(e)
    int split_tokens;          // keys per split, multiple of 64
    int max_splits;            // ceil(max_blocks * block_size / split_tokens)
    float *ws_o;               // [B * Hq * max_splits, 128] partial outputs
    float *ws_lse;             // [B * Hq * max_splits] log2-sum-exp of each split
    int *err_count;
};

// Keys per split for given sizes (kv_split_tokens 0 = automatic).
int decode_resolve_split(int B, int Hkv, int max_blocks, int block_size, int kv_split_tokens,
                         int num_sms);
size_t decode_workspace_bytes(int B, int Hq, int max_splits);

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, cudaStream_t s);

// The host-side argument checks of nv_decode_attn_paged (everything but the
// workspace and the memory kind of the caches) and its split plan.  Returns
// NV_OK (plan filled; all zero when B == 0) or the NV_E* code the entry point
// returns for these arguments.
struct DecodePlan {
    int split_tokens;          // keys per split
    int max_splits;            // splits of the longest context the table allows
    size_t workspace_bytes;    // workspace the call needs (0: none)
};
int decode_check_args(const void *q, int64_t q_tok_stride, const void *k_cache,
                      const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, const void *o, int B, int Hq, int Hkv,
                      int head_dim, int block_size, int64_t num_blocks, float softmax_scale,
                      int kv_split_tokens, DecodePlan *plan);

// True for device or managed memory (what the tensor-memory accelerator can
// read); false for host memory or a pointer the runtime does not know.
bool device_addressable_for_tma(const void *p);

// ----------------------------------------------------------------- prefill
struct PrefillParams {
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_k;
    uint16_t *o;
    int B, Hq, Hkv;
    int max_seqlen_q;
    float scale_log2;
    int *err_count;
    int *work_counter;         // optional: items handed out by atomicAdd (cleared per launch)
    // Paged K/V only: keys come from the cache through the block table.
    const int32_t *block_tables;
    int max_blocks;
    int block_size;            // multiple of 128
    int64_t num_blocks;
};

// paged == false: k/v maps are 3-D [128, Hkv, total_k] over contiguous k/v;
// paged == true: 4-D [128, Hkv, block_size, num_blocks] over the caches.
cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map, bool paged,
                           cudaStream_t s);

// --------------------------------------------------------------------- TMA
// Build a bf16 tiled tensor map with 128-byte swizzling (the innermost box
// dimension must be 64 elements).  dims/strides are innermost first; strides
// are in bytes for dims 1..rank-1.  Returns false on failure.
bool make_tensor_map_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box);

}  // namespace nvattn
