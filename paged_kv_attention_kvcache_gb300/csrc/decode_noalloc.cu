// nv_decode_attn_paged_noalloc: paged decode attention for callers that are
// handed only their input and output buffers and cannot allocate device
// memory themselves -- for example a plugin running inside a host framework
// that owns every device allocation, or a serving loop that has committed all
// free HBM to its KV-cache pool and may not call cudaMalloc while serving.
//
// The split-KV workspace that nv_decode_attn_paged takes from its caller
// lives here instead, in one file-scope device array of fixed size that
// every GPU loading this library keeps until the process exits.  The decode
// itself is the unchanged nv_decode_attn_paged path, given that array.
#include <mutex>

#include "../../include/nv_attn.h"

namespace {

constexpr size_t kScratchBytes = NV_DECODE_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code this name is only a host-side stand-in
// for the symbol, not a device address; the device address is looked up
// with cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up the
// first time this device is seen.  Returns nullptr on failure.
void *scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();   // do not leave the error for a later launch check
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" NV_API int nv_decode_attn_paged_noalloc(
    const nv_bf16_t *q, int64_t q_tok_stride, const nv_bf16_t *k_cache,
    const nv_bf16_t *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, nv_bf16_t *o, int B, int Hq, int Hkv, int head_dim,
    int block_size, int64_t num_blocks, float softmax_scale, int kv_split_tokens,
    int *err_count, void *stream) {
    const bool sizes_ok = B > 0 && Hq > 0 && Hkv > 0 && head_dim == 128 &&
                          max_blocks_per_seq > 0 && block_size > 0 && kv_split_tokens >= 0;
    size_t need = 0;
    if (sizes_ok) {
        need = nv_decode_attn_workspace_size(B, Hq, Hkv, head_dim, max_blocks_per_seq,
                                             block_size, kv_split_tokens);
        if (need > kScratchBytes) return NV_EWORKSPACE;    // beyond the fixed scratch
    }
    if (!sizes_ok || need == 0)
        // Nothing to stage in the scratch array: either the arguments are
        // rejected (or B == 0) by the regular entry point, or every sequence
        // fits in one split and no workspace is used.
        return nv_decode_attn_paged(q, q_tok_stride, k_cache, v_cache, block_tables,
                                    max_blocks_per_seq, context_lens, o, B, Hq, Hkv, head_dim,
                                    block_size, num_blocks, softmax_scale, kv_split_tokens,
                                    nullptr, 0, err_count, stream);
    void *scratch = scratch_for_current_device();
    if (!scratch) return NV_ELAUNCH;
    // Every workspace slot the merge kernel reads is first written by the
    // split kernel of the same call, so nothing here needs clearing.
    return nv_decode_attn_paged(q, q_tok_stride, k_cache, v_cache, block_tables,
                                max_blocks_per_seq, context_lens, o, B, Hq, Hkv, head_dim,
                                block_size, num_blocks, softmax_scale, kv_split_tokens,
                                scratch, kScratchBytes, err_count, stream);
}
