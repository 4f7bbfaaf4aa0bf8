/*
 * Reference oracle for the Qwen3 attention-sublayer hot path (nano-vllm).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke check
 * in __graft_entry__ and the CPU-baseline leg of bench.py may load this file.
 * It shares no code, header, helper or table with the CUDA library; the two
 * meet only on the seeded inputs produced by the `workloads` package.
 *
 * Every function is the plain definition of what the method computes, written
 * in fp64 with no tiling, no fusion and no reordering beyond the definition.
 * bf16 inputs are widened exactly (a bf16 value is the top 16 bits of an
 * IEEE fp32 value).  Outputs are fp64 unless the operation is a byte copy.
 *
 * Sources (page title, then section):
 *   [RMS]   "3.3 Model skeleton and core operators", sec. 2 RMSNorm
 *           (rms_forward / add_rms_forward); and "同一个 Qwen3，两种写法",
 *           sec. 3.6 (the fused residual add).
 *   [ROPE]  "3.3 Model skeleton and core operators", sec. 3 RoPE (inv_freq,
 *           half-split rotation); "同一个 Qwen3，两种写法", sec. 2 config
 *           (rope_theta 1e6) and sec. 3.5.
 *   [QKN]   "3.3 Model skeleton and core operators", sec. 8 (q_norm/k_norm
 *           over head_dim, before rotary_emb); "Nano-vLLM 源码解读 第17篇",
 *           sec. 4 QK-Norm 与 RoPE.
 *   [STORE] "3.3 Model skeleton and core operators", sec. 7.1;
 *           "Nano-vLLM 源码解读 第17篇", sec. 5.1 store_kvcache.
 *   [ATTN]  "3.3 Model skeleton and core operators", sec. 7.2 (scale
 *           head_dim^-0.5, causal=True); "Nano-vLLM 源码解读 第17篇",
 *           sec. 5.2 FlashAttention (tiling is an exact rearrangement of
 *           softmax(QK^T * scale) V); "同一个 Qwen3，两种写法", sec. 3.2
 *           (packed varlen layout, block-diagonal causal mask) and sec. 3.4
 *           (GQA handled inside the kernel, no repeat_kv).
 *   [SWIGLU] "3.3 Model skeleton and core operators", sec. 4 SwiGLU:
 *           SiluAndMul (gate first, up second) and sec. 5 (Qwen3MLP).
 *   [PAGED] "nano-vllm code walkthrough", Prefill stage case 2 and Decode
 *           Stage (block_table "stitches" physical blocks into the logical
 *           K/V sequence; cache_seqlens = current length of each sequence).
 *
 * Where the pages are silent, the reading taken is stated at the function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the upper half of an fp32. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Round fp64 values to bf16 bit patterns, round-to-nearest-even.  The pages
 * keep every activation and the KV cache in the model dtype, bfloat16
 * ("同一个 Qwen3，两种写法", sec. 2 config: torch_dtype bfloat16); the oracle
 * uses this only where a chained flow stores a bf16 tensor (q/k after RoPE,
 * the cache).  Finite inputs only.
 */
void orc_round_to_bf16(const double *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        double x = in[i];
        double ax = fabs(x);
        uint16_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x8000u : 0u;
        if (ax == 0.0) { out[i] = sign; continue; }
        int e;
        /* ax = m * 2^e with m in [0.5, 1) */
        double m = frexp(ax, &e);
        /* bf16 normal numbers: value = 1.f * 2^(E-127), 7 fraction bits.
           Work with an integer significand of 8 bits: sig in [128, 256). */
        int exp2 = e - 1;            /* ax = (2m) * 2^exp2, 2m in [1,2) */
        if (exp2 < -126) {           /* subnormal range: fixed quantum 2^-133 */
            double q = ldexp(ax, 133);
            double r = nearbyint(q); /* default rounding mode: nearest-even */
            uint32_t mant = (uint32_t)r;           /* may reach 128 = min normal */
            out[i] = (uint16_t)(sign | mant);
            continue;
        }
        double scaled = ldexp(m, 8);              /* in [128, 256) */
        double r = nearbyint(scaled);             /* nearest-even */
        uint32_t sig = (uint32_t)r;
        if (sig == 256) { sig = 128; exp2 += 1; }
        if (exp2 > 127) { out[i] = (uint16_t)(sign | 0x7F80u); continue; } /* inf */
        uint32_t biased = (uint32_t)(exp2 + 127);
        out[i] = (uint16_t)(sign | (biased << 7) | (sig - 128));
    }
}

/*
 * [RMS] Residual-add RMSNorm, one row of H features at a time:
 *   s = x + residual          (the pages add in fp32; here exactly, in fp64)
 *   residual_out = s          (the new residual is the sum itself)
 *   y = s / sqrt(mean(s^2) + eps) * weight
 * With residual == NULL it is the plain RMSNorm of x and residual_out is not
 * written.  The norm uses the unrounded sum (the pages compute the variance
 * from the fp32 sum, not from the bf16 copy they return).
 */
int orc_add_rmsnorm(const uint16_t *x, const uint16_t *residual,
                    const uint16_t *weight, int64_t T, int64_t H, double eps,
                    double *y, double *residual_out) {
    if (T < 0 || H <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *s = (double *)malloc((size_t)H * sizeof(double));
        double sum_sq = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            double v = bf16_bits_to_double(x[t * H + i]);
            if (residual) v += bf16_bits_to_double(residual[t * H + i]);
            s[i] = v;
            sum_sq += v * v;
        }
        double mean_sq = sum_sq / (double)H;
        double inv_rms = 1.0 / sqrt(mean_sq + eps);
        for (int64_t i = 0; i < H; ++i) {
            y[t * H + i] = s[i] * inv_rms * bf16_bits_to_double(weight[i]);
            if (residual && residual_out) residual_out[t * H + i] = s[i];
        }
        free(s);
    }
    return 0;
}

/*
 * [ROPE] The rotary table as the pages define it, evaluated exactly:
 *   inv_freq[i] = 1 / base^(2i / rotary_dim),  i = 0 .. rotary_dim/2 - 1
 *   angle(p, i) = p * inv_freq[i]
 *   row p = [cos(angle(p, 0..)), sin(angle(p, 0..))]      (cos half, sin half)
 * The pages build it in fp32; the oracle keeps the exact fp64 angle.
 */
int orc_rope_cos_sin(int64_t max_position, int rotary_dim, double base,
                     double *cos_sin) {
    if (max_position < 0 || rotary_dim <= 0 || (rotary_dim & 1)) return -1;
    int half = rotary_dim / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < max_position; ++p) {
        for (int i = 0; i < half; ++i) {
            double inv_freq = 1.0 / pow(base, (double)(2 * i) / (double)rotary_dim);
            double angle = (double)p * inv_freq;
            cos_sin[p * rotary_dim + i] = cos(angle);
            cos_sin[p * rotary_dim + half + i] = sin(angle);
        }
    }
    return 0;
}

/*
 * [QKN] + [ROPE] Per-head RMSNorm over head_dim followed by the half-split
 * rotation, for one projection (q or k) at a time:
 *   n = x / sqrt(mean(x^2) + eps) * w                 (w: q_norm or k_norm)
 *   for i < d/2:  y[i]       = n[i] cos(a_i) - n[i+d/2] sin(a_i)
 *                 y[i+d/2]   = n[i+d/2] cos(a_i) + n[i] sin(a_i)
 *   with a_i = positions[t] * base^(-2i/d).
 * x is [T, nheads, d] with token stride tok_stride (elements) and heads
 * contiguous; out is [T, nheads, d] contiguous.  eps is the model's
 * rms_norm_eps (the pages never show the q_norm constructor).
 */
int orc_qknorm_rope(const uint16_t *x, int64_t tok_stride, int64_t T,
                    int nheads, int d, const uint16_t *w,
                    const int64_t *positions, double base, double eps,
                    double *out) {
    if (T < 0 || nheads <= 0 || d <= 0 || (d & 1)) return -1;
    int half = d / 2;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double *n = (double *)malloc((size_t)d * sizeof(double));
        double pos = (double)positions[t];
        for (int h = 0; h < nheads; ++h) {
            const uint16_t *row = x + t * tok_stride + (int64_t)h * d;
            double sum_sq = 0.0;
            for (int i = 0; i < d; ++i) {
                double v = bf16_bits_to_double(row[i]);
                sum_sq += v * v;
            }
            double inv_rms = 1.0 / sqrt(sum_sq / (double)d + eps);
            for (int i = 0; i < d; ++i)
                n[i] = bf16_bits_to_double(row[i]) * inv_rms * bf16_bits_to_double(w[i]);
            double *o = out + (t * nheads + h) * (int64_t)d;
            for (int i = 0; i < half; ++i) {
                double inv_freq = 1.0 / pow(base, (double)(2 * i) / (double)d);
                double a = pos * inv_freq;
                double c = cos(a), s = sin(a);
                o[i] = n[i] * c - n[i + half] * s;
                o[i + half] = n[i + half] * c + n[i] * s;
            }
        }
        free(n);
    }
    return 0;
}

/*
 * [STORE] For every token n whose slot is not -1, copy its D = Hkv*d key
 * elements to row `slot` of the flat cache view [num_slots, D], and likewise
 * for the value.  slot == -1 marks a padding token and writes nothing.  Any
 * other slot outside [0, num_slots) is not defined by the pages; it is
 * skipped and counted, and the count is returned.
 */
int64_t orc_store_kvcache(const uint16_t *key, int64_t key_stride,
                          const uint16_t *value, int64_t value_stride,
                          uint16_t *k_cache, uint16_t *v_cache,
                          const int32_t *slot_mapping, int64_t N, int64_t D,
                          int64_t num_slots) {
    int64_t bad = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) { ++bad; continue; }
        memcpy(k_cache + slot * D, key + n * key_stride, (size_t)D * sizeof(uint16_t));
        memcpy(v_cache + slot * D, value + n * value_stride, (size_t)D * sizeof(uint16_t));
    }
    return bad;
}

/*
 * [SWIGLU] SiluAndMul: row t of x holds 2*I values, the first I the gate g
 * and the last I the up projection u (the merged gate_up output, split in
 * half along the last dim, gate first).  out[t][i] = silu(g_i) * u_i with
 * silu(g) = g / (1 + exp(-g)).  The pages run it under torch.compile, which
 * fuses the two ops; the plain reading is one value per element, rounded
 * once at the end, so it is returned unrounded here.
 */
int orc_silu_and_mul(const uint16_t *x, int64_t x_stride, int64_t T, int64_t I, double *out) {
    if (T < 0 || I < 0 || x_stride < 2 * I) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < I; ++i) {
            double g = bf16_bits_to_double(x[t * x_stride + i]);
            double u = bf16_bits_to_double(x[t * x_stride + I + i]);
            out[t * I + i] = g / (1.0 + exp(-g)) * u;
        }
    }
    return 0;
}

/*
 * Dense softmax attention of one query row over L keys (the definition):
 *   s_j = scale * <q, k_j>;  p_j = exp(s_j - max s) / sum_j exp(s_j - max s)
 *   o   = sum_j p_j v_j
 * k_rows[j] / v_rows[j] point at the d elements of key/value j.  L == 0
 * gives o = 0.
 */
static void dense_attention_row(const double *q, const uint16_t *const *k_rows,
                                const uint16_t *const *v_rows, int64_t L, int d,
                                double scale, double *scores, double *o) {
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (L <= 0) return;
    double m = -INFINITY;
    for (int64_t j = 0; j < L; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += q[i] * bf16_bits_to_double(k_rows[j][i]);
        scores[j] = scale * acc;
        if (scores[j] > m) m = scores[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < L; ++j) {
        scores[j] = exp(scores[j] - m);
        denom += scores[j];
    }
    for (int64_t j = 0; j < L; ++j) {
        double p = scores[j] / denom;
        for (int i = 0; i < d; ++i) o[i] += p * bf16_bits_to_double(v_rows[j][i]);
    }
}

/*
 * [ATTN] Varlen attention over packed sequences.  Sequence b owns query
 * tokens [cu_q[b], cu_q[b+1]) and key tokens [cu_k[b], cu_k[b+1]).  Query
 * head h reads kv head h / (Hq/Hkv).  With causal != 0, query i of a
 * sequence with Lq queries and Lk keys sees keys j <= i + (Lk - Lq): for
 * Lq == Lk that is j <= i; for Lk > Lq the mask is aligned to the last key
 * (the bottom-right alignment used for prefix-cache prefill).  No mask
 * crosses a sequence boundary.
 *
 * q/k/v are [tokens, heads, d] with the given token strides (elements),
 * heads contiguous.  If rows == NULL, every (token, head) is computed and out
 * is [Tq, Hq, d]; otherwise rows holds n_rows (token, head) pairs and out is
 * [n_rows, d].
 */
int orc_attention_varlen(const uint16_t *q, int64_t q_stride,
                         const uint16_t *k, int64_t k_stride,
                         const uint16_t *v, int64_t v_stride,
                         const int32_t *cu_q, const int32_t *cu_k, int B,
                         int Hq, int Hkv, int d, double scale, int causal,
                         const int64_t *rows, int64_t n_rows, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0) return -1;
    int group = Hq / Hkv;
    int64_t Tq = B > 0 ? cu_q[B] : 0;
    int64_t n_units = rows ? n_rows : Tq * Hq;
    int64_t max_lk = 0;
    for (int b = 0; b < B; ++b) {
        int64_t lk = (int64_t)cu_k[b + 1] - cu_k[b];
        if (lk > max_lk) max_lk = lk;
    }
    int status = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc((size_t)(max_lk > 0 ? max_lk : 1) * sizeof(double));
        const uint16_t **k_rows = (const uint16_t **)malloc((size_t)(max_lk > 0 ? max_lk : 1) * sizeof(void *));
        const uint16_t **v_rows = (const uint16_t **)malloc((size_t)(max_lk > 0 ? max_lk : 1) * sizeof(void *));
        double *qv = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t u = 0; u < n_units; ++u) {
            int64_t t = rows ? rows[2 * u] : u / Hq;
            int h = rows ? (int)rows[2 * u + 1] : (int)(u % Hq);
            double *o = out + u * d;
            int b = -1;
            for (int s = 0; s < B; ++s)
                if (t >= cu_q[s] && t < cu_q[s + 1]) { b = s; break; }
            if (b < 0 || h < 0 || h >= Hq) {
                for (int i = 0; i < d; ++i) o[i] = NAN;
#pragma omp atomic write
                status = -2;
                continue;
            }
            int64_t i_q = t - cu_q[b];
            int64_t lq = (int64_t)cu_q[b + 1] - cu_q[b];
            int64_t lk = (int64_t)cu_k[b + 1] - cu_k[b];
            int64_t visible = lk;
            if (causal) {
                visible = i_q + (lk - lq) + 1;
                if (visible > lk) visible = lk;
                if (visible < 0) visible = 0;
            }
            int kvh = h / group;
            for (int64_t j = 0; j < visible; ++j) {
                int64_t tok = cu_k[b] + j;
                k_rows[j] = k + tok * k_stride + (int64_t)kvh * d;
                v_rows[j] = v + tok * v_stride + (int64_t)kvh * d;
            }
            const uint16_t *qrow = q + t * q_stride + (int64_t)h * d;
            for (int i = 0; i < d; ++i) qv[i] = bf16_bits_to_double(qrow[i]);
            dense_attention_row(qv, k_rows, v_rows, visible, d, scale, scores, o);
        }
        free(scores); free(k_rows); free(v_rows); free(qv);
    }
    return status;
}

/*
 * [PAGED] Single-query decode over a paged cache.  For sequence b the
 * logical K (and V) sequence of length L = context_lens[b] is stitched
 * together block by block: logical token j lives in physical block
 * block_tables[b][j / block_size] at offset j % block_size.  The stitched
 * copy is then fed to the dense definition; the single query sees all L
 * keys (causality with one query aligned to the last key masks nothing).
 * The cache is [num_blocks, block_size, Hkv, d]; q is [B, Hq, d] with token
 * stride q_stride; out is [B, Hq, d] (pairs == NULL) or [n_pairs, d] for the
 * listed (b, h) pairs.  Returns -3 if a block id needed by some L is outside
 * [0, num_blocks) or L exceeds max_blocks * block_size.
 */
int orc_paged_decode(const uint16_t *q, int64_t q_stride,
                     const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_tables, int max_blocks,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int d,
                     int block_size, int64_t num_blocks, double scale,
                     const int64_t *pairs, int64_t n_pairs, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || block_size <= 0) return -1;
    int group = Hq / Hkv;
    int64_t n_units = pairs ? n_pairs : (int64_t)B * Hq;
    int64_t max_l = (int64_t)max_blocks * block_size;
    int status = 0;
#pragma omp parallel
    {
        /* The stitched logical sequence for one (b, kv head). */
        uint16_t *k_seq = (uint16_t *)malloc((size_t)(max_l > 0 ? max_l : 1) * d * sizeof(uint16_t));
        uint16_t *v_seq = (uint16_t *)malloc((size_t)(max_l > 0 ? max_l : 1) * d * sizeof(uint16_t));
        const uint16_t **k_rows = (const uint16_t **)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(void *));
        const uint16_t **v_rows = (const uint16_t **)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(void *));
        double *scores = (double *)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(double));
        double *qv = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < n_units; ++u) {
            int b = pairs ? (int)pairs[2 * u] : (int)(u / Hq);
            int h = pairs ? (int)pairs[2 * u + 1] : (int)(u % Hq);
            double *o = out + u * d;
            int64_t L = context_lens[b];
            if (L < 0 || L > max_l) {
                for (int i = 0; i < d; ++i) o[i] = NAN;
#pragma omp atomic write
                status = -3;
                continue;
            }
            int kvh = h / group;
            int ok = 1;
            for (int64_t j = 0; j < L; ++j) {
                int64_t blk = block_tables[(int64_t)b * max_blocks + j / block_size];
                if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
                int64_t off = ((blk * block_size + j % block_size) * Hkv + kvh) * (int64_t)d;
                memcpy(k_seq + j * d, k_cache + off, (size_t)d * sizeof(uint16_t));
                memcpy(v_seq + j * d, v_cache + off, (size_t)d * sizeof(uint16_t));
                k_rows[j] = k_seq + j * d;
                v_rows[j] = v_seq + j * d;
            }
            if (!ok) {
                for (int i = 0; i < d; ++i) o[i] = NAN;
#pragma omp atomic write
                status = -3;
                continue;
            }
            const uint16_t *qrow = q + (int64_t)b * q_stride + (int64_t)h * d;
            for (int i = 0; i < d; ++i) qv[i] = bf16_bits_to_double(qrow[i]);
            dense_attention_row(qv, k_rows, v_rows, L, d, scale, scores, o);
        }
        free(k_seq); free(v_seq); free(k_rows); free(v_rows); free(scores); free(qv);
    }
    return status;
}

/*
 * [PAGED] + [ATTN] Prefill over the paged cache: a prefix-cache hit or a
 * later chunk of chunked prefill ("3.3 Model skeleton and core operators",
 * sec. 7.2: k, v are replaced by the whole cache and block_table is passed;
 * "nano-vllm code walkthrough", Prefill stage case 2).  Sequence b has
 * Lq = cu_q[b+1] - cu_q[b] new queries and Lk = cu_k[b+1] - cu_k[b] keys in
 * the cache (prefix plus the new tokens, already stored); its logical K/V
 * sequence is stitched block by block through block_tables[b].  Query i sits
 * at position Lk - Lq + i and sees keys j <= Lk - Lq + i (causality aligned
 * to the last key).  q is [Tq, Hq, d] with token stride q_stride; out is
 * [Tq, Hq, d] (rows == NULL) or [n_rows, d].  Returns -3 on a block id
 * outside [0, num_blocks) or Lk > max_blocks * block_size, -4 if Lk < Lq.
 */
int orc_attention_paged_prefill(const uint16_t *q, int64_t q_stride,
                                const uint16_t *k_cache, const uint16_t *v_cache,
                                const int32_t *block_tables, int max_blocks,
                                const int32_t *cu_q, const int32_t *cu_k, int B,
                                int Hq, int Hkv, int d, int block_size,
                                int64_t num_blocks, double scale,
                                const int64_t *rows, int64_t n_rows, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || block_size <= 0) return -1;
    int group = Hq / Hkv;
    int64_t Tq = B > 0 ? cu_q[B] : 0;
    int64_t n_units = rows ? n_rows : Tq * Hq;
    int64_t max_l = (int64_t)max_blocks * block_size;
    int status = 0;
#pragma omp parallel
    {
        uint16_t *k_seq = (uint16_t *)malloc((size_t)(max_l > 0 ? max_l : 1) * d * sizeof(uint16_t));
        uint16_t *v_seq = (uint16_t *)malloc((size_t)(max_l > 0 ? max_l : 1) * d * sizeof(uint16_t));
        const uint16_t **k_rows = (const uint16_t **)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(void *));
        const uint16_t **v_rows = (const uint16_t **)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(void *));
        double *scores = (double *)malloc((size_t)(max_l > 0 ? max_l : 1) * sizeof(double));
        double *qv = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < n_units; ++u) {
            int64_t t = rows ? rows[2 * u] : u / Hq;
            int h = rows ? (int)rows[2 * u + 1] : (int)(u % Hq);
            double *o = out + u * d;
            int b = -1;
            for (int s = 0; s < B; ++s)
                if (t >= cu_q[s] && t < cu_q[s + 1]) { b = s; break; }
            int64_t lq = b >= 0 ? (int64_t)cu_q[b + 1] - cu_q[b] : 0;
            int64_t lk = b >= 0 ? (int64_t)cu_k[b + 1] - cu_k[b] : 0;
            int bad = b < 0 || h < 0 || h >= Hq ? -2 : (lk > max_l ? -3 : (lk < lq ? -4 : 0));
            if (bad) {
                for (int i = 0; i < d; ++i) o[i] = NAN;
#pragma omp atomic write
                status = bad;
                continue;
            }
            int64_t i_q = t - cu_q[b];
            int64_t visible = i_q + (lk - lq) + 1;
            int kvh = h / group;
            int ok = 1;
            for (int64_t j = 0; j < visible; ++j) {
                int64_t blk = block_tables[(int64_t)b * max_blocks + j / block_size];
                if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
                int64_t off = ((blk * block_size + j % block_size) * Hkv + kvh) * (int64_t)d;
                memcpy(k_seq + j * d, k_cache + off, (size_t)d * sizeof(uint16_t));
                memcpy(v_seq + j * d, v_cache + off, (size_t)d * sizeof(uint16_t));
                k_rows[j] = k_seq + j * d;
                v_rows[j] = v_seq + j * d;
            }
            if (!ok) {
                for (int i = 0; i < d; ++i) o[i] = NAN;
#pragma omp atomic write
                status = -3;
                continue;
            }
            const uint16_t *qrow = q + t * q_stride + (int64_t)h * d;
            for (int i = 0; i < d; ++i) qv[i] = bf16_bits_to_double(qrow[i]);
            dense_attention_row(qv, k_rows, v_rows, visible, d, scale, scores, o);
        }
        free(k_seq); free(v_seq); free(k_rows); free(v_rows); free(scores); free(qv);
    }
    return status;
}
