// extern "C" entry points of libnvattn.so (declared in include/nv_attn.h).
// Each one checks its arguments on the host, builds any TMA descriptors the
// kernels need, and launches on the caller's stream.  Nothing here allocates,
// synchronises or copies device memory.
#include <math.h>
#include <mutex>

#include "../../include/nv_attn.h"
#include "internal.h"

namespace nvattn {

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensors read through TMA must be device (or managed) memory; pinned host
// memory is fine only for the tensors the kernels touch with plain loads and
// stores.  A host pointer here would make the tensor copy fault, so it is
// rejected before anything is launched.
bool tma_readable(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // do not leave the error for a later launch check
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? NV_OK : NV_ELAUNCH; }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library links only the static CUDA runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int num_sms_current_device() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return 152;
    return sms;
}

}  // namespace

bool make_tensor_map_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank) gstride[i] = strides_bytes[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                    const_cast<void *>(base), gdim, gstride, bdim, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int decode_check_args(const void *q, int64_t q_tok_stride, const void *k_cache,
                      const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, const void *o, int B, int Hq, int Hkv,
                      int head_dim, int block_size, int64_t num_blocks, float softmax_scale,
                      int kv_split_tokens, DecodePlan *plan) {
    plan->split_tokens = 0;
    plan->max_splits = 0;
    plan->workspace_bytes = 0;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq <= 0 ||
        block_size <= 0 || num_blocks <= 0 || kv_split_tokens < 0 || !(softmax_scale > 0.f) ||
        !isfinite(softmax_scale))
        return NV_EINVAL;
    if (head_dim != 128 || block_size % 64 != 0 || Hq / Hkv > 16 || B > 65535 || Hkv > 65535)
        return NV_EUNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > 0x7FFFFFFF || num_blocks > 0x7FFFFFFF)
        return NV_EUNSUPPORTED;
    if (B == 0) return NV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !o) return NV_EINVAL;
    if (q_tok_stride < (int64_t)Hq * 128) return NV_EINVAL;
    if (q_tok_stride % 8 || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(o))
        return NV_EALIGN;
    const int split = decode_resolve_split(B, Hkv, max_blocks_per_seq, block_size,
                                           kv_split_tokens, num_sms_current_device());
    const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
    const int max_splits = (int)((max_ctx + split - 1) / split);
    if (max_splits > 65535) return NV_EUNSUPPORTED;
    plan->split_tokens = split;
    plan->max_splits = max_splits;
    plan->workspace_bytes = decode_workspace_bytes(B, Hq, max_splits);
    return NV_OK;
}

bool device_addressable_for_tma(const void *p) { return tma_readable(p); }

}  // namespace nvattn

using namespace nvattn;

extern "C" {

const char *nv_status_string(int status) {
    switch (status) {
        case NV_OK: return "NV_OK";
        case NV_EINVAL: return "NV_EINVAL: invalid argument";
        case NV_EUNSUPPORTED: return "NV_EUNSUPPORTED: unsupported shape";
        case NV_EALIGN: return "NV_EALIGN: pointer or stride not 16-byte aligned";
        case NV_EWORKSPACE: return "NV_EWORKSPACE: workspace missing or too small";
        case NV_ELAUNCH: return "NV_ELAUNCH: kernel launch failed";
        case NV_EDRIVER: return "NV_EDRIVER: TMA descriptor could not be built";
        default: return "unknown status";
    }
}

int nv_version(void) { return 100; }

int nv_rope_cos_sin_cache(float *cos_sin, int max_position, int rotary_dim, double base,
                          void *stream) {
    if (max_position < 0 || rotary_dim <= 0 || (rotary_dim & 1) || rotary_dim > 1024 ||
        !(base > 1.0) || !isfinite(base))
        return NV_EINVAL;
    if (max_position == 0) return NV_OK;
    if (!cos_sin) return NV_EINVAL;
    return launch_status(launch_rope_cos_sin(cos_sin, max_position, rotary_dim, base,
                                             as_stream(stream)));
}

int nv_add_rmsnorm(const nv_bf16_t *x, const nv_bf16_t *residual, const nv_bf16_t *weight,
                   nv_bf16_t *out, nv_bf16_t *residual_out, int64_t T, int H,
                   int64_t row_stride, float eps, void *stream) {
    if (T < 0 || T > 0x7FFFFFFF || H <= 0 || row_stride < H || !(eps >= 0.f) || !isfinite(eps))
        return NV_EINVAL;
    if (H % 8 != 0 || H > 16384) return NV_EUNSUPPORTED;
    if (T == 0) return NV_OK;
    if (!x || !weight || !out || (residual && !residual_out)) return NV_EINVAL;
    if (row_stride % 8 || !aligned16(x) || !aligned16(weight) || !aligned16(out) ||
        (residual && (!aligned16(residual) || !aligned16(residual_out))))
        return NV_EALIGN;
    return launch_status(launch_add_rmsnorm(x, residual, weight, out,
                                            residual ? residual_out : nullptr, T, H, row_stride,
                                            eps, as_stream(stream)));
}

int nv_qknorm_rope(nv_bf16_t *q, int64_t q_tok_stride, nv_bf16_t *k, int64_t k_tok_stride,
                   const nv_bf16_t *q_norm_weight, const nv_bf16_t *k_norm_weight,
                   const float *cos_sin, int max_position, const int64_t *positions, int64_t T,
                   int Hq, int Hkv, int head_dim, float eps, int *err_count, void *stream) {
    if (T < 0 || Hq <= 0 || Hkv <= 0 || max_position <= 0 || !(eps >= 0.f) || !isfinite(eps))
        return NV_EINVAL;
    if (head_dim != 128) return NV_EUNSUPPORTED;
    if (T == 0) return NV_OK;
    if (!q || !k || !q_norm_weight || !k_norm_weight || !cos_sin || !positions)
        return NV_EINVAL;
    if (q_tok_stride < (int64_t)Hq * 128 || k_tok_stride < (int64_t)Hkv * 128) return NV_EINVAL;
    if (q_tok_stride % 8 || k_tok_stride % 8 || !aligned16(q) || !aligned16(k) ||
        !aligned16(q_norm_weight) || !aligned16(k_norm_weight) || !aligned16(cos_sin))
        return NV_EALIGN;
    if (T * (int64_t)(Hq + Hkv) * 8 > (int64_t)0x7FFFFFFF * 256) return NV_EUNSUPPORTED;
    return launch_status(launch_qknorm_rope(q, q_tok_stride, k, k_tok_stride, q_norm_weight,
                                            k_norm_weight, cos_sin, max_position, positions, T,
                                            Hq, Hkv, eps, err_count, as_stream(stream)));
}

int nv_store_kvcache(const nv_bf16_t *key, int64_t key_tok_stride, const nv_bf16_t *value,
                     int64_t value_tok_stride, nv_bf16_t *k_cache, nv_bf16_t *v_cache,
                     const int32_t *slot_mapping, int64_t N, int Hkv, int head_dim,
                     int64_t num_slots, int *err_count, void *stream) {
    if (N < 0 || Hkv <= 0 || head_dim <= 0 || num_slots < 0) return NV_EINVAL;
    const int64_t D = (int64_t)Hkv * head_dim;
    if (D % 8 != 0 || D > 8192) return NV_EUNSUPPORTED;
    if (N == 0) return NV_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return NV_EINVAL;
    if (key_tok_stride < D || value_tok_stride < D) return NV_EINVAL;
    if (key_tok_stride % 8 || value_tok_stride % 8 || !aligned16(key) || !aligned16(value) ||
        !aligned16(k_cache) || !aligned16(v_cache))
        return NV_EALIGN;
    return launch_status(launch_store_kvcache(key, key_tok_stride, value, value_tok_stride,
                                              k_cache, v_cache, slot_mapping, N, (int)D,
                                              num_slots, err_count, as_stream(stream)));
}

int nv_qknorm_rope_store(nv_bf16_t *q, int64_t q_tok_stride, nv_bf16_t *k,
                         int64_t k_tok_stride, const nv_bf16_t *v, int64_t v_tok_stride,
                         const nv_bf16_t *q_norm_weight, const nv_bf16_t *k_norm_weight,
                         const float *cos_sin, int max_position, const int64_t *positions,
                         const int32_t *slot_mapping, nv_bf16_t *k_cache, nv_bf16_t *v_cache,
                         int64_t num_slots, int64_t T, int Hq, int Hkv, int head_dim, float eps,
                         int write_k, int *err_count, void *stream) {
    if (T < 0 || Hq <= 0 || Hkv <= 0 || max_position <= 0 || num_slots < 0 ||
        !(eps >= 0.f) || !isfinite(eps) || (write_k != 0 && write_k != 1))
        return NV_EINVAL;
    if (head_dim != 128) return NV_EUNSUPPORTED;
    if (T == 0) return NV_OK;
    if (!q || !k || !v || !q_norm_weight || !k_norm_weight || !cos_sin || !positions ||
        !slot_mapping || !k_cache || !v_cache)
        return NV_EINVAL;
    if (q_tok_stride < (int64_t)Hq * 128 || k_tok_stride < (int64_t)Hkv * 128 ||
        v_tok_stride < (int64_t)Hkv * 128)
        return NV_EINVAL;
    if (q_tok_stride % 8 || k_tok_stride % 8 || v_tok_stride % 8 || !aligned16(q) ||
        !aligned16(k) || !aligned16(v) || !aligned16(q_norm_weight) ||
        !aligned16(k_norm_weight) || !aligned16(cos_sin) || !aligned16(k_cache) ||
        !aligned16(v_cache))
        return NV_EALIGN;
    if (T * (int64_t)(Hq + 2 * Hkv) * 8 > (int64_t)0x7FFFFFFF * 256) return NV_EUNSUPPORTED;
    return launch_status(launch_qknorm_rope_store(
        q, q_tok_stride, k, k_tok_stride, v, v_tok_stride, q_norm_weight, k_norm_weight, cos_sin,
        max_position, positions, slot_mapping, k_cache, v_cache, num_slots, T, Hq, Hkv, eps,
        write_k, err_count, as_stream(stream)));
}

int nv_selftest_wait_timeout(int *err_count, void *stream) {
    if (!err_count || (uintptr_t)err_count % 4) return NV_EINVAL;
    return launch_status(launch_wait_timeout_selftest(err_count, as_stream(stream)));
}

int nv_silu_and_mul(const nv_bf16_t *x, int64_t x_tok_stride, nv_bf16_t *out,
                    int64_t out_tok_stride, int64_t T, int intermediate, void *stream) {
    if (T < 0 || intermediate < 0) return NV_EINVAL;
    if (intermediate % 8) return NV_EUNSUPPORTED;
    if (T == 0 || intermediate == 0) return NV_OK;
    if (!x || !out) return NV_EINVAL;
    if (x_tok_stride < 2 * (int64_t)intermediate || out_tok_stride < intermediate)
        return NV_EINVAL;
    if (x_tok_stride % 8 || out_tok_stride % 8 || !aligned16(x) || !aligned16(out))
        return NV_EALIGN;
    // The only overlap allowed is out == x with the same token stride.
    const uintptr_t x0 = (uintptr_t)x, o0 = (uintptr_t)out;
    const uintptr_t x1 = x0 + (uintptr_t)(((T - 1) * x_tok_stride + 2 * (int64_t)intermediate) * 2);
    const uintptr_t o1 = o0 + (uintptr_t)(((T - 1) * out_tok_stride + intermediate) * 2);
    const bool overlap = x0 < o1 && o0 < x1;
    if (overlap && !(o0 == x0 && out_tok_stride == x_tok_stride)) return NV_EINVAL;
    return launch_status(launch_silu_and_mul(x, x_tok_stride, out, out_tok_stride, T,
                                             intermediate, as_stream(stream)));
}

int nv_prefill_attn_varlen(const nv_bf16_t *q, int64_t q_tok_stride, const nv_bf16_t *k,
                           int64_t k_tok_stride, const nv_bf16_t *v, int64_t v_tok_stride,
                           nv_bf16_t *o, const int32_t *cu_seqlens_q,
                           const int32_t *cu_seqlens_k, int B, int64_t total_q, int64_t total_k,
                           int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int head_dim,
                           float softmax_scale, int causal, int *sched_counter, int *err_count,
                           void *stream) {
    if (B < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !(softmax_scale > 0.f) || !isfinite(softmax_scale))
        return NV_EINVAL;
    if (head_dim != 128 || causal != 1) return NV_EUNSUPPORTED;
    if (total_q >= 0x7FFFFFFF || total_k >= 0x7FFFFFFF || B > 65535 || Hq > 65535)
        return NV_EUNSUPPORTED;
    if (B == 0 || total_q == 0 || max_seqlen_q == 0) return NV_OK;
    if (!q || !k || !v || !o || !cu_seqlens_q || !cu_seqlens_k) return NV_EINVAL;
    if (q_tok_stride < (int64_t)Hq * 128 || k_tok_stride < (int64_t)Hkv * 128 ||
        v_tok_stride < (int64_t)Hkv * 128)
        return NV_EINVAL;
    if (q_tok_stride % 8 || k_tok_stride % 8 || v_tok_stride % 8 || !aligned16(q) ||
        !aligned16(k) || !aligned16(v) || !aligned16(o) || ((uintptr_t)sched_counter & 3))
        return NV_EALIGN;
    if ((int64_t)(max_seqlen_q + 127) / 128 > 65535) return NV_EUNSUPPORTED;
    if (!tma_readable(q) || !tma_readable(k) || !tma_readable(v)) return NV_EINVAL;

    CUtensorMap q_map, k_map, v_map;
    const uint32_t box[3] = {64, 1, 128};
    {
        const uint64_t dims[3] = {128, (uint64_t)Hq, (uint64_t)total_q};
        const uint64_t strides[2] = {128 * 2, (uint64_t)q_tok_stride * 2};
        if (!make_tensor_map_bf16(&q_map, q, 3, dims, strides, box)) return NV_EDRIVER;
    }
    {
        const uint64_t dims[3] = {128, (uint64_t)Hkv, (uint64_t)(total_k > 0 ? total_k : 1)};
        uint64_t strides[2] = {128 * 2, (uint64_t)k_tok_stride * 2};
        if (!make_tensor_map_bf16(&k_map, k, 3, dims, strides, box)) return NV_EDRIVER;
        strides[1] = (uint64_t)v_tok_stride * 2;
        if (!make_tensor_map_bf16(&v_map, v, 3, dims, strides, box)) return NV_EDRIVER;
    }
    PrefillParams p;
    p.cu_seqlens_q = cu_seqlens_q;
    p.cu_seqlens_k = cu_seqlens_k;
    p.o = o;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.max_seqlen_q = max_seqlen_q;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.err_count = err_count;
    p.work_counter = sched_counter;
    p.block_tables = nullptr;
    p.max_blocks = 0;
    p.block_size = 0;
    p.num_blocks = 0;
    return launch_status(launch_prefill(p, q_map, k_map, v_map, false, as_stream(stream)));
}

int nv_prefill_attn_paged(const nv_bf16_t *q, int64_t q_tok_stride, const nv_bf16_t *k_cache,
                          const nv_bf16_t *v_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, nv_bf16_t *o, const int32_t *cu_seqlens_q,
                          const int32_t *cu_seqlens_k, int B, int64_t total_q, int max_seqlen_q,
                          int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
                          float softmax_scale, int causal, int *sched_counter, int *err_count,
                          void *stream) {
    if (B < 0 || total_q < 0 || max_seqlen_q < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 ||
        max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 ||
        !(softmax_scale > 0.f) || !isfinite(softmax_scale))
        return NV_EINVAL;
    if (head_dim != 128 || causal != 1 || block_size % 128 != 0) return NV_EUNSUPPORTED;
    if (total_q >= 0x7FFFFFFF || B > 65535 || Hq > 65535 || num_blocks > 0x7FFFFFFF ||
        (int64_t)max_blocks_per_seq * block_size > 0x7FFFFFFF)
        return NV_EUNSUPPORTED;
    if (B == 0 || total_q == 0 || max_seqlen_q == 0) return NV_OK;
    if (!q || !k_cache || !v_cache || !o || !block_tables || !cu_seqlens_q || !cu_seqlens_k)
        return NV_EINVAL;
    if (q_tok_stride < (int64_t)Hq * 128) return NV_EINVAL;
    if (q_tok_stride % 8 || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(o) || ((uintptr_t)sched_counter & 3))
        return NV_EALIGN;
    if ((int64_t)(max_seqlen_q + 127) / 128 > 65535) return NV_EUNSUPPORTED;
    if (!tma_readable(q) || !tma_readable(k_cache) || !tma_readable(v_cache)) return NV_EINVAL;

    CUtensorMap q_map, k_map, v_map;
    {
        const uint64_t dims[3] = {128, (uint64_t)Hq, (uint64_t)total_q};
        const uint64_t strides[2] = {128 * 2, (uint64_t)q_tok_stride * 2};
        const uint32_t box[3] = {64, 1, 128};
        if (!make_tensor_map_bf16(&q_map, q, 3, dims, strides, box)) return NV_EDRIVER;
    }
    {
        const uint64_t dims[4] = {128, (uint64_t)Hkv, (uint64_t)block_size, (uint64_t)num_blocks};
        const uint64_t strides[3] = {128 * 2, (uint64_t)Hkv * 128 * 2,
                                     (uint64_t)block_size * Hkv * 128 * 2};
        const uint32_t box[4] = {64, 1, 128, 1};
        if (!make_tensor_map_bf16(&k_map, k_cache, 4, dims, strides, box) ||
            !make_tensor_map_bf16(&v_map, v_cache, 4, dims, strides, box))
            return NV_EDRIVER;
    }
    PrefillParams p;
    p.cu_seqlens_q = cu_seqlens_q;
    p.cu_seqlens_k = cu_seqlens_k;
    p.o = o;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.max_seqlen_q = max_seqlen_q;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.err_count = err_count;
    p.work_counter = sched_counter;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    return launch_status(launch_prefill(p, q_map, k_map, v_map, true, as_stream(stream)));
}

size_t nv_decode_attn_workspace_size(int B, int Hq, int Hkv, int head_dim,
                                     int max_blocks_per_seq, int block_size,
                                     int kv_split_tokens) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || head_dim != 128 || max_blocks_per_seq <= 0 ||
        block_size <= 0 || kv_split_tokens < 0)
        return 0;
    const int split = decode_resolve_split(B, Hkv, max_blocks_per_seq, block_size,
                                           kv_split_tokens, num_sms_current_device());
    const int64_t max_ctx = (int64_t)max_blocks_per_seq * block_size;
    const int max_splits = (int)((max_ctx + split - 1) / split);
    return decode_workspace_bytes(B, Hq, max_splits);
}

int nv_decode_attn_paged(const nv_bf16_t *q, int64_t q_tok_stride, const nv_bf16_t *k_cache,
                         const nv_bf16_t *v_cache, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *context_lens, nv_bf16_t *o,
                         int B, int Hq, int Hkv, int head_dim, int block_size,
                         int64_t num_blocks, float softmax_scale, int kv_split_tokens,
                         void *workspace, size_t workspace_bytes, int *err_count,
                         void *stream) {
    DecodePlan plan;
    const int st = decode_check_args(q, q_tok_stride, k_cache, v_cache, block_tables,
                                     max_blocks_per_seq, context_lens, o, B, Hq, Hkv, head_dim,
                                     block_size, num_blocks, softmax_scale, kv_split_tokens,
                                     &plan);
    if (st != NV_OK || B == 0) return st;
    const int split = plan.split_tokens;
    const int max_splits = plan.max_splits;
    const size_t need = plan.workspace_bytes;
    if (need > 0 && (!workspace || workspace_bytes < need)) return NV_EWORKSPACE;
    if (need > 0 && !aligned16(workspace)) return NV_EALIGN;
    if (!tma_readable(k_cache) || !tma_readable(v_cache)) return NV_EINVAL;

    CUtensorMap k_map, v_map;
    const uint64_t dims[4] = {128, (uint64_t)Hkv, (uint64_t)block_size, (uint64_t)num_blocks};
    const uint64_t strides[3] = {128 * 2, (uint64_t)Hkv * 128 * 2,
                                 (uint64_t)block_size * Hkv * 128 * 2};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (!make_tensor_map_bf16(&k_map, k_cache, 4, dims, strides, box) ||
        !make_tensor_map_bf16(&v_map, v_cache, 4, dims, strides, box))
        return NV_EDRIVER;

    DecodeParams p;
    p.q = q;
    p.q_stride = q_tok_stride;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.o = o;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.split_tokens = split;
    p.max_splits = max_splits;
    const size_t n = (size_t)B * Hq * max_splits;
    p.ws_o = need ? static_cast<float *>(workspace) : nullptr;
    p.ws_lse = need ? static_cast<float *>(workspace) + n * 128 : nullptr;
    p.err_count = err_count;
    return launch_status(launch_decode(p, k_map, v_map, as_stream(stream)));
}

}  // extern "C"
