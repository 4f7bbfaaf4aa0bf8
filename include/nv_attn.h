/*
 * nv_attn.h — C ABI of libnvattn.so: the device work of one Qwen3 attention
 * sublayer as nano-vllm runs it, written for NVIDIA GB300 (sm_103a).
 *
 * Operations, in the order one layer calls them:
 *   nv_add_rmsnorm          fused residual add + RMSNorm (input_layernorm)
 *   nv_qknorm_rope          per-head RMSNorm of q and k, then RoPE, in place
 *   nv_store_kvcache        scatter new K/V rows into the paged cache
 *   nv_qknorm_rope_store    the two above in one pass (k goes straight to its slot)
 *   nv_prefill_attn_varlen  causal GQA attention over packed sequences
 *   nv_prefill_attn_paged   the same with K/V read through the block table
 *   nv_decode_attn_paged    single-query GQA attention over the paged cache
 *   nv_silu_and_mul         the MLP's SwiGLU activation that follows the sublayer
 * plus nv_rope_cos_sin_cache (builds the RoPE table once) and the decode
 * workspace query.
 *
 * Conventions shared by every entry point
 *   - Every tensor is caller-owned memory the device can address: device
 *     memory (allocated e.g. by PyTorch), or, for the tensors the kernels
 *     touch only with ordinary loads and stores, pinned host memory mapped
 *     into the device's address space (cudaHostAlloc / cudaHostRegister with
 *     unified addressing, as on Grace-Blackwell), which the kernels then read
 *     and write over the host link.  Tensors read through the tensor-memory
 *     accelerator must be device (or managed) memory: the KV caches of
 *     nv_decode_attn_paged and nv_prefill_attn_paged, and q, k, v of
 *     nv_prefill_attn_varlen (q of nv_prefill_attn_paged too); these calls
 *     return NV_EINVAL for anything else.  Everything else may be either.
 *     The library never allocates, frees, synchronises or reads results
 *     back; every call only enqueues kernels on `stream` (a cudaStream_t;
 *     NULL means the legacy default stream) and returns.
 *   - bf16 tensors are passed as `nv_bf16_t` (the 16 raw bits of a bfloat16).
 *     Integer metadata is int32 (slot_mapping, block_tables, context_lens,
 *     cu_seqlens) except positions, which are int64, as in nano-vllm.
 *   - Strides are in ELEMENTS.  Within a token, heads are contiguous and
 *     head_dim is contiguous (stride 1), matching the views nano-vllm makes
 *     of its packed qkv buffer.
 *   - Return value: NV_OK (0) or a negative NV_E* code.  Arguments are
 *     checked on the host before anything is launched; on any error nothing
 *     is launched and device memory is untouched.  NV_ELAUNCH reports a
 *     failed launch (cudaGetLastError after the launch).
 *   - Device-side index faults that the host cannot see (a slot, block id,
 *     context length or position out of range) never trap: the element is
 *     skipped and, if `err_count` is non-NULL, atomically counted there.
 *   - No entry point waits on another CTA.  Waits inside a CTA (its own
 *     copy and tensor-core pipeline) give up after about a second; the
 *     kernel then sets bit 30 (NV_ERR_PIPELINE_FAILURE) of err_count, leaves
 *     the affected outputs unwritten (decode writes NaN into them instead)
 *     and finishes.  CTAs that start after the bit is set skip their work.
 *     Only a defect can cause this; clear err_count before reusing it.
 *   - Calls are asynchronous and allocate nothing.
 *
 * Sources are cited by page title and section.
 */
#ifndef NV_ATTN_H
#define NV_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define NV_API __attribute__((visibility("default")))
#else
#define NV_API
#endif

typedef uint16_t nv_bf16_t;

#define NV_OK            0
#define NV_EINVAL       -1  /* null pointer, negative or inconsistent size  */
#define NV_EUNSUPPORTED -2  /* shape outside what the kernels implement     */
#define NV_EALIGN       -3  /* pointer or stride not 16-byte aligned        */
#define NV_EWORKSPACE   -4  /* decode workspace missing or too small        */
#define NV_ELAUNCH      -5  /* kernel launch failed                          */
#define NV_EDRIVER      -6  /* TMA descriptor could not be built            */

/* Bit of *err_count set when an in-kernel pipeline wait gave up. */
#define NV_ERR_PIPELINE_FAILURE (1 << 30)

/* Human-readable name of a status code (static string). */
NV_API const char *nv_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
NV_API int nv_version(void);

/*
 * RoPE table.  "3.3 Model skeleton and core operators", sec. 3: cos and sin
 * of position * inv_freq, inv_freq[i] = 1 / base^(2i / rotary_dim), stored
 * as one row per position, cos half then sin half.
 *   cos_sin      [max_position, rotary_dim] fp32, written.
 *   base         rope_theta (1e6 for Qwen3).
 * The angle is formed in fp64 on the device and only the result is rounded
 * to fp32 (the pages form it in fp32; at position 40959 that costs up to
 * ~2e-3 rad, which this table avoids).  rotary_dim must be even, <= 1024.
 */
NV_API int nv_rope_cos_sin_cache(float *cos_sin, int max_position, int rotary_dim,
                          double base, void *stream);

/*
 * Fused residual add + RMSNorm.  "3.3 Model skeleton and core operators",
 * sec. 2 (add_rms_forward / rms_forward); "同一个 Qwen3，两种写法", sec. 3.6.
 * Per row t of H features:
 *   s = x + residual (fp32);  residual_out = bf16(s);
 *   out = bf16(s * rsqrt(mean(s^2) + eps) * weight)
 * residual == NULL gives the plain RMSNorm of x (first layer); residual_out
 * is then not written and may be NULL.
 *   x, residual, out, residual_out   [T, H] bf16; row t of each starts
 *                                    row_stride elements after row t - 1
 *                                    (row_stride == H: contiguous rows).
 *   weight                           [H] bf16 (gamma).
 * residual_out may alias residual (in place); out may alias x.  Other
 * overlaps are undefined.  Requires H % 8 == 0, 8 <= H <= 16384,
 * row_stride >= H and a multiple of 8, all pointers 16-byte aligned.
 * T == 0 is a no-op.
 */
NV_API int nv_add_rmsnorm(const nv_bf16_t *x, const nv_bf16_t *residual,
                   const nv_bf16_t *weight, nv_bf16_t *out,
                   nv_bf16_t *residual_out, int64_t T, int H,
                   int64_t row_stride, float eps, void *stream);

/*
 * QK-Norm + RoPE, in place.  "3.3 Model skeleton and core operators",
 * sec. 8 (q_norm / k_norm over head_dim when qkv_bias is false, then
 * rotary_emb) and sec. 3 (half-split rotation: dimension i pairs with
 * i + head_dim/2); "Nano-vLLM 源码解读 第17篇", sec. 4.
 * For each token t and head h of q (weight q_norm_weight) and of k
 * (weight k_norm_weight):
 *   n = x * rsqrt(mean(x^2) + eps) * w                  (fp32)
 *   x[i]       <- bf16(n[i] * cos - n[i+64] * sin)
 *   x[i + 64]  <- bf16(n[i+64] * cos + n[i] * sin)      (i < 64)
 * with (cos, sin) = cos_sin[positions[t]].  V is never touched.
 *   q            [T, Hq, head_dim] bf16, token stride q_tok_stride.
 *   k            [T, Hkv, head_dim] bf16, token stride k_tok_stride.
 *   cos_sin      [max_position, head_dim] fp32 (nv_rope_cos_sin_cache).
 *   positions    [T] int64.
 * A position outside [0, max_position) leaves that token's q and k
 * unchanged and is counted in err_count.  Requires head_dim == 128,
 * token strides multiples of 8, pointers 16-byte aligned.
 */
NV_API int nv_qknorm_rope(nv_bf16_t *q, int64_t q_tok_stride, nv_bf16_t *k,
                   int64_t k_tok_stride, const nv_bf16_t *q_norm_weight,
                   const nv_bf16_t *k_norm_weight, const float *cos_sin,
                   int max_position, const int64_t *positions, int64_t T,
                   int Hq, int Hkv, int head_dim, float eps, int *err_count,
                   void *stream);

/*
 * store_kvcache.  "3.3 Model skeleton and core operators", sec. 7.1;
 * "Nano-vLLM 源码解读 第17篇", sec. 5.1.  For every token n with
 * slot_mapping[n] != -1, copy its D = Hkv * head_dim key elements to row
 * slot_mapping[n] of the cache viewed as [num_slots, D], and likewise the
 * value.  A bit copy: the cache receives exactly the input bits.
 *   key, value        [N, Hkv, head_dim] bf16, token strides key_tok_stride,
 *                     value_tok_stride (heads contiguous).
 *   k_cache, v_cache  [num_blocks, block_size, Hkv, head_dim] bf16,
 *                     num_slots = num_blocks * block_size.
 *   slot_mapping      [N] int32 (-1 = padding, skipped silently).
 * Any other slot outside [0, num_slots) is skipped and counted.  Requires
 * D % 8 == 0, D <= 8192, strides multiples of 8, 16-byte aligned pointers.
 * Two tokens naming the same slot leave one of them there (unspecified
 * which).
 */
NV_API int nv_store_kvcache(const nv_bf16_t *key, int64_t key_tok_stride,
                     const nv_bf16_t *value, int64_t value_tok_stride,
                     nv_bf16_t *k_cache, nv_bf16_t *v_cache,
                     const int32_t *slot_mapping, int64_t N, int Hkv,
                     int head_dim, int64_t num_slots, int *err_count,
                     void *stream);

/*
 * QK-Norm + RoPE + store_kvcache in one pass.  "Nano-vLLM 源码解读 第17篇",
 * sec. 4 and 5.1, and "3.3 Model skeleton and core operators", sec. 7.1 and
 * 8: the attention forward rotates q and k and then scatters k and v into
 * the paged cache; this call does both steps per token, so the rotated k
 * goes from registers straight to its cache slot.  For in-range positions
 * the result is exactly that of nv_qknorm_rope followed by
 * nv_store_kvcache on the same arguments, bit for bit, except that k in
 * place is written only when
 * write_k == 1 (the contiguous prefill reads it there; decode and the
 * paged prefill read the cache and pass write_k == 0).
 *   q, k, v      [T, Hq|Hkv|Hkv, head_dim] bf16 views, token strides as given;
 *                q is rotated in place, v is only read.
 *   q_norm_weight, k_norm_weight, cos_sin, positions, eps   as nv_qknorm_rope.
 *   slot_mapping [T] int32; -1 = padding (nothing cached for that token).
 *   k_cache, v_cache [num_blocks, block_size, Hkv, head_dim] bf16,
 *                num_slots = num_blocks * block_size.
 * A slot outside [0, num_slots) other than -1 is counted once per token and
 * the token's rows are not cached; a position outside [0, max_position) is
 * counted per q and k row as in nv_qknorm_rope, and leaves q, k and the
 * token's k cache row untouched (its v row is still copied).  Requires
 * head_dim == 128, token strides multiples of 8, 16-byte aligned pointers.
 * T == 0 is a no-op.  No counterpart in nano-vllm, which runs the two steps
 * as separate kernels; it is a design variant of the same step order.
 */
NV_API int nv_qknorm_rope_store(nv_bf16_t *q, int64_t q_tok_stride, nv_bf16_t *k,
                                int64_t k_tok_stride, const nv_bf16_t *v,
                                int64_t v_tok_stride, const nv_bf16_t *q_norm_weight,
                                const nv_bf16_t *k_norm_weight, const float *cos_sin,
                                int max_position, const int64_t *positions,
                                const int32_t *slot_mapping, nv_bf16_t *k_cache,
                                nv_bf16_t *v_cache, int64_t num_slots, int64_t T, int Hq,
                                int Hkv, int head_dim, float eps, int write_k,
                                int *err_count, void *stream);

/*
 * Failure-path self-test (no page counterpart: it checks this library's own
 * stall reporting).  Launches one CTA whose thread waits on a shared-memory
 * mbarrier that nothing arrives on, through the same bounded wait every
 * pipeline here uses.  The wait gives up after about a second and sets
 * NV_ERR_PIPELINE_FAILURE in *err_count, as a stalled pipeline would; the
 * kernel then exits normally, so the context stays usable.  Later calls that
 * are given the same err_count skip their work while the bit is set (clear
 * it first).
 *   err_count    one int the device can address (4-byte aligned), required.
 * Returns NV_EINVAL for a null or misaligned err_count.
 */
NV_API int nv_selftest_wait_timeout(int *err_count, void *stream);

/*
 * SiluAndMul, the SwiGLU activation of the MLP that follows the attention
 * sublayer.  "3.3 Model skeleton and core operators", sec. 4 (SwiGLU:
 * SiluAndMul splits the merged gate_up output in half along the last dim,
 * gate first) and sec. 5 (Qwen3MLP: gate_up_proj -> act_fn -> down_proj).
 * With I = intermediate:
 *   out[t][i] = bf16( silu(x[t][i]) * x[t][I + i] ),  silu(g) = g / (1 + e^-g)
 * in fp32 with one rounding at the end (the pages run it under
 * torch.compile, which fuses the two ops).
 *   x    [T, 2I] bf16, token stride x_tok_stride (>= 2I).
 *   out  [T, I] bf16, token stride out_tok_stride (>= I), written.
 * out may equal x when the two strides are equal (the result then fills the
 * gate half); any other overlap is rejected with NV_EINVAL.  Requires
 * I % 8 == 0, strides multiples of 8, 16-byte aligned pointers.  T == 0 or
 * I == 0 is a no-op.
 */
NV_API int nv_silu_and_mul(const nv_bf16_t *x, int64_t x_tok_stride, nv_bf16_t *out,
                           int64_t out_tok_stride, int64_t T, int intermediate,
                           void *stream);

/*
 * Varlen causal prefill attention.  "3.3 Model skeleton and core
 * operators", sec. 7.2 (flash_attn_varlen_func, scale head_dim^-0.5,
 * causal=True); "同一个 Qwen3，两种写法", sec. 3.2 (packed [T, ...] layout,
 * cu_seqlens boundaries, block-diagonal causal mask); "nano-vllm code
 * walkthrough", Prefill stage case 1 (contiguous k/v, q and k lengths equal).
 * For sequence b (queries [cu_seqlens_q[b], cu_seqlens_q[b+1]), keys
 * [cu_seqlens_k[b], cu_seqlens_k[b+1])), query head h and query row i:
 *   o = sum_{j <= i} softmax_j(softmax_scale * <q_i, k_j>) v_j
 * with k, v taken from kv head h / (Hq / Hkv).  Computed on tcgen05 tensor
 * cores: bf16 operands, fp32 accumulation in tensor memory, fp32 softmax.
 *   q      [total_q, Hq, head_dim] bf16, token stride q_tok_stride.
 *   k, v   [total_k, Hkv, head_dim] bf16, token strides k_/v_tok_stride.
 *   o      [total_q, Hq, head_dim] bf16, contiguous, written.
 *   cu_seqlens_q, cu_seqlens_k   [B + 1] int32, device.
 *   max_seqlen_q, max_seqlen_k   upper bounds of the per-sequence lengths
 *                                (they size the grid; larger is safe).
 * Causality is aligned to the last key: with Lq queries and Lk keys in a
 * sequence, query i sees keys j <= Lk - Lq + i, so equal lengths give the
 * plain prefill and Lk > Lq a prefill whose first Lk - Lq keys are an
 * earlier prefix.  Requires causal == 1 and Lk >= Lq for every sequence (a
 * sequence with Lk < Lq is skipped and counted in err_count).  Rows of other
 * sequences that share a 128-row tile are read but masked, and V rows past a
 * sequence's last key are zeroed in shared memory before use, so another
 * sequence's rows may hold any bits (NaN included) without reaching o.
 * Requires head_dim == 128, token strides multiples of 8, 16-byte aligned
 * pointers, total_q, total_k < 2^31.  err_count (optional) counts skipped
 * sequences and records NV_ERR_PIPELINE_FAILURE.
 * sched_counter (optional, recommended): one int of device memory, 4-byte
 * aligned, through which the persistent CTAs draw work items heaviest first
 * (an atomic counter), which balances ragged batches.  The call clears it
 * with an enqueued memset before its kernel, so its contents on entry do
 * not matter, but calls that may run concurrently need distinct counters.
 * NULL gives a fixed round-robin assignment of items to CTAs.
 */
NV_API int nv_prefill_attn_varlen(const nv_bf16_t *q, int64_t q_tok_stride,
                           const nv_bf16_t *k, int64_t k_tok_stride,
                           const nv_bf16_t *v, int64_t v_tok_stride,
                           nv_bf16_t *o, const int32_t *cu_seqlens_q,
                           const int32_t *cu_seqlens_k, int B, int64_t total_q,
                           int64_t total_k, int max_seqlen_q, int max_seqlen_k,
                           int Hq, int Hkv, int head_dim, float softmax_scale,
                           int causal, int *sched_counter, int *err_count,
                           void *stream);

/*
 * Prefill over the paged cache: a prefix-cache hit, or a later chunk of a
 * chunked prefill.  "3.3 Model skeleton and core operators", sec. 7.2 (when
 * K/V of the step already sit in the cache, k and v are replaced by the
 * whole k_cache / v_cache and block_table is passed; cu_seqlens_k[-1] >
 * cu_seqlens_q[-1]); "nano-vllm code walkthrough", Prefill stage case 2.
 * Sequence b has Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b] new queries and
 * Lk = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys, all already in the cache
 * (nv_store_kvcache wrote the new ones first); logical key j lives at
 * k_cache[block_tables[b][j / block_size], j % block_size, h / G].  Query i
 * sees keys j <= Lk - Lq + i.  Same tcgen05 kernel as
 * nv_prefill_attn_varlen, with K/V tiles gathered through the block table.
 *   q             [total_q, Hq, head_dim] bf16, token stride q_tok_stride.
 *   k_cache, v_cache  [num_blocks, block_size, Hkv, head_dim] bf16.
 *   block_tables  [B, max_blocks_per_seq] int32.
 *   o             [total_q, Hq, head_dim] bf16, contiguous, written.
 * A block id outside [0, num_blocks) is counted in err_count and reads as
 * zeros; a sequence with Lk < Lq or Lk > max_blocks_per_seq * block_size is
 * skipped and counted.  Cache rows past Lk may hold any bits.  Requires
 * head_dim == 128, block_size % 128 == 0, causal == 1, 16-byte aligned
 * pointers, q_tok_stride a multiple of 8.  sched_counter as for
 * nv_prefill_attn_varlen.
 */
NV_API int nv_prefill_attn_paged(const nv_bf16_t *q, int64_t q_tok_stride,
                                 const nv_bf16_t *k_cache, const nv_bf16_t *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 nv_bf16_t *o, const int32_t *cu_seqlens_q,
                                 const int32_t *cu_seqlens_k, int B, int64_t total_q,
                                 int max_seqlen_q, int Hq, int Hkv, int head_dim,
                                 int block_size, int64_t num_blocks, float softmax_scale,
                                 int causal, int *sched_counter, int *err_count,
                                 void *stream);

/*
 * Bytes of fp32 workspace nv_decode_attn_paged needs for these sizes and
 * this kv_split_tokens (0 = automatic, resolved exactly as the decode call
 * resolves it on the current device).  Returns 0 when no workspace is
 * needed and also on invalid sizes.
 */
NV_API size_t nv_decode_attn_workspace_size(int B, int Hq, int Hkv, int head_dim,
                                     int max_blocks_per_seq, int block_size,
                                     int kv_split_tokens);

/*
 * Paged decode attention.  "3.3 Model skeleton and core operators", sec. 7.2
 * (flash_attn_with_kvcache with cache_seqlens = context_lens and
 * block_table); "nano-vllm code walkthrough", Decode Stage; split-KV with a
 * log-sum-exp merge is the rescaling identity of "Nano-vLLM 源码解读 第17篇",
 * sec. 5.2 applied across key ranges.
 * For sequence b and query head h, with L = context_lens[b] (it counts the
 * token just written by nv_store_kvcache):
 *   o[b, h] = sum_{j < L} softmax_j(softmax_scale * <q[b,h], K_j>) V_j,
 *   K_j = k_cache[block_tables[b][j / block_size], j % block_size, h / G]
 * with G = Hq / Hkv (same for V).  L == 0 writes zeros.
 *   q             [B, Hq, head_dim] bf16, token stride q_tok_stride.
 *   k_cache, v_cache  [num_blocks, block_size, Hkv, head_dim] bf16.
 *   block_tables  [B, max_blocks_per_seq] int32 (entries past
 *                 ceil(L / block_size) are never read; -1 padding is fine).
 *   context_lens  [B] int32.
 *   o             [B, Hq, head_dim] bf16, contiguous, written.
 *   kv_split_tokens  keys per split (rounded up to a multiple of 64);
 *                 0 = automatic: chosen from B, Hkv, the longest context
 *                 (max_blocks_per_seq * block_size) and the SM count,
 *                 usually 1024-4096 keys, 512 for a very small grid; short
 *                 contexts over many sequences are not split at all.  A
 *                 sequence longer than one split is
 *                 processed by several CTAs whose partial (O, log-sum-exp)
 *                 go to `workspace` and are merged by a second kernel.
 *   workspace     device buffer of at least
 *                 nv_decode_attn_workspace_size(...) bytes (may be NULL
 *                 when that size is 0); contents on entry are ignored.
 * A block id outside [0, num_blocks) or L > max_blocks_per_seq *
 * block_size is counted in err_count; the offending keys are skipped: o is
 * the attention over the keys that remain, zeros if none remain.
 * Requires head_dim == 128, block_size % 64 == 0, 1 <= G <= 16, 16-byte
 * aligned pointers, q_tok_stride a multiple of 8, B <= 65535.
 */
NV_API int nv_decode_attn_paged(const nv_bf16_t *q, int64_t q_tok_stride,
                         const nv_bf16_t *k_cache, const nv_bf16_t *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, nv_bf16_t *o, int B,
                         int Hq, int Hkv, int head_dim, int block_size,
                         int64_t num_blocks, float softmax_scale,
                         int kv_split_tokens, void *workspace,
                         size_t workspace_bytes, int *err_count, void *stream);

/*
 * Paged decode attention that allocates nothing and takes no workspace.
 * The paper has no counterpart: it exists for callers that are handed only
 * their input and output buffers and cannot allocate device memory -- a
 * plugin inside a host framework that owns every allocation, or a serving
 * loop that has committed all free HBM to its KV cache and may not call
 * cudaMalloc while serving.
 *
 * Arguments and results are those of nv_decode_attn_paged without
 * `workspace` / `workspace_bytes`.  The split-KV partial results go to one
 * library-owned device array of NV_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB),
 * which every GPU that loads the library holds until the process exits.
 *   - Returns NV_EWORKSPACE, launching nothing, when these sizes would need
 *     more than that (nv_decode_attn_workspace_size(...) with the same
 *     arguments tells in advance); use nv_decode_attn_paged, a larger
 *     kv_split_tokens, or fewer sequences per call.
 *   - Arguments are checked exactly as nv_decode_attn_paged checks them,
 *     with the same codes; NV_EWORKSPACE comes only for a call that is
 *     otherwise valid.
 *   - The first call on each device looks up the array's device address
 *     with that device current (and looks it up again when the device's
 *     context has changed, e.g. after cudaDeviceReset); make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero: every slot the merge reads was
 *     written by the same call, and after a pipeline failure the merge reads
 *     none).  Calls whose kernels overlap on the GPU -- on different
 *     streams, or from different threads -- race on it; serialise them.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define NV_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

NV_API int nv_decode_attn_paged_noalloc(const nv_bf16_t *q, int64_t q_tok_stride,
                                        const nv_bf16_t *k_cache,
                                        const nv_bf16_t *v_cache,
                                        const int32_t *block_tables,
                                        int max_blocks_per_seq,
                                        const int32_t *context_lens, nv_bf16_t *o,
                                        int B, int Hq, int Hkv, int head_dim,
                                        int block_size, int64_t num_blocks,
                                        float softmax_scale, int kv_split_tokens,
                                        int *err_count, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* NV_ATTN_H */
