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
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = NV_DECODE_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code this name is only a host-side stand-in
// for the symbol, not a device address; the device address is looked up
// with cudaGetSymbolAddress below, once per device (and context).
static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;

struct ScratchEntry {
    CUcontext ctx;   // context the address belongs to
    void *ptr;       // device address of g_decode_scratch in that context
};

std::mutex g_lock;
ScratchEntry g_scratch[kMaxDevices] = {};

// cuCtxGetCurrent, fetched from the driver through the runtime (the library
// links only the static CUDA runtime).  nullptr if unavailable.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current() {
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

CUcontext current_context() {
    CtxGetCurrentFn fn = ctx_get_current();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the scratch array on the current device, looked up the
// first time this device is seen and again whenever the device's current
// context is not the one the address was taken in (cudaDeviceReset replaces
// the primary context and reloads the module).  Returns nullptr on failure.
void *scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> guard(g_lock);
    const CUcontext ctx = current_context();
    ScratchEntry &e = g_scratch[dev];
    if (e.ptr && ctx && e.ctx == ctx) return e.ptr;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();   // do not leave the error for a later launch check
        return nullptr;
    }
    // The lookup makes the device's primary context current if none was.
    e.ctx = ctx ? ctx : current_context();
    e.ptr = ptr;
    return ptr;
}

}  // namespace

extern "C" NV_API int nv_decode_attn_paged_noalloc(
    const nv_bf16_t *q, int64_t q_tok_stride, const nv_bf16_t *k_cache,
    const nv_bf16_t *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, nv_bf16_t *o, int B, int Hq, int Hkv, int head_dim,
    int block_size, int64_t num_blocks, float softmax_scale, int kv_split_tokens,
    int *err_count, void *stream) {
    // The regular entry point's checks come first, so that a call it would
    // reject gets the same code here; only a valid call can be too large
    // for the fixed scratch array.
    nvattn::DecodePlan plan;
    const int st = nvattn::decode_check_args(q, q_tok_stride, k_cache, v_cache, block_tables,
                                             max_blocks_per_seq, context_lens, o, B, Hq, Hkv,
                                             head_dim, block_size, num_blocks, softmax_scale,
                                             kv_split_tokens, &plan);
    if (st != NV_OK || B == 0) return st;
    if (!nvattn::device_addressable_for_tma(k_cache) ||
        !nvattn::device_addressable_for_tma(v_cache))
        return NV_EINVAL;
    if (plan.workspace_bytes > kScratchBytes) return NV_EWORKSPACE;   // beyond the fixed array
    void *scratch = nullptr;
    if (plan.workspace_bytes > 0) {
        scratch = scratch_for_current_device();
        if (!scratch) return NV_ELAUNCH;
    }
    // A split writes its workspace slots before the merge reads them; after a
    // pipeline failure (bit 30 of err_count) the merge reads none, and a split
    // whose wait gave up writes NaN, so an earlier call's partials never
    // reach o.  Nothing in the array needs clearing.
    return nv_decode_attn_paged(q, q_tok_stride, k_cache, v_cache, block_tables,
                                max_blocks_per_seq, context_lens, o, B, Hq, Hkv, head_dim,
                                block_size, num_blocks, softmax_scale, kv_split_tokens,
                                scratch, scratch ? kScratchBytes : 0, err_count, stream);
}
