// Paged single-query decode attention with split-KV and a log-sum-exp merge.
//
// What it computes ("3.3 Model skeleton and core operators", sec. 7.2;
// "nano-vllm code walkthrough", Decode Stage): for sequence b and query head
// h, softmax(scale * q K^T) V over the first context_lens[b] tokens of the
// logical sequence that block_tables[b] stitches out of the paged cache, K
// and V taken from kv head h / G.
//
// How (GB300):
//  - One CTA per (split, kv head, sequence).  A split is a run of
//    `split_tokens` keys; all G = Hq / Hkv query heads of the kv head live in
//    the CTA, so every K/V byte is read from HBM exactly once.
//  - A producer warp walks the block table and issues 4-D TMA loads of
//    64-token tiles (two 128-byte-swizzled halves of head_dim for K and for
//    V, 32 KB per stage) into a ring of shared-memory stages guarded by
//    mbarriers.
//  - Four consumer warps each take 16 tokens of a tile.  The G query rows
//    (padded to 16) form the A operand of mma.m16n8k16 for S = Q K^T and the
//    bf16 probabilities are reused in registers as the A operand of O += P V;
//    K and V fragments come from the swizzled tiles through ldmatrix.  Softmax
//    is online (running max m, denominator l, output O) in fp32, base 2.
//  - The four warps' (m, l, O) are combined in shared memory.  A sequence
//    that fits in one split writes bf16 output directly; otherwise each split
//    writes its normalised partial output and log2-sum-exp to the workspace
//    and decode_merge_kernel combines them: with M = max_s lse_s,
//    O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).  This is the exact
//    rescaling identity of "Nano-vLLM 源码解读 第17篇", sec. 5.2, applied
//    across key ranges.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace nvattn {

constexpr int kTile = 64;                         // tokens per pipeline stage
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 1);
constexpr int kHalfTileBytes = kTile * 64 * 2;    // 64 tokens x 64 dims bf16
constexpr int kStageBytes = 4 * kHalfTileBytes;   // K lo, K hi, V lo, V hi
constexpr int kCombStride = 132;                  // padded fp32 row (bank spread)
constexpr int kDecodeSmemBytes = kStages * kStageBytes + 1024 + 2 * kStages * 8;

static_assert(kConsumerWarps * 16 == kTile, "each consumer warp owns 16 tokens of a tile");
static_assert(kConsumerWarps * 16 * kCombStride * 4 + 2 * kConsumerWarps * 16 * 4 <=
                  kStages * kStageBytes,
              "warp-combine scratch must fit in the stage buffers");

__device__ __forceinline__ void named_barrier_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
    pdl_wait_release();
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;
    const int max_l = p.max_blocks * p.block_size;
    int L = __ldg(p.context_lens + b);
    if (L < 0 || L > max_l) {
        if (split == 0 && g == 0 && threadIdx.x == 0) count_error(p.err_count);
        L = L < 0 ? 0 : max_l;
    }
    const int64_t head0 = (int64_t)b * p.Hq + (int64_t)g * G;   // first query head of the group
    if (L == 0) {
        if (split == 0) {
            for (int idx = threadIdx.x; idx < G * 128; idx += kDecodeThreads)
                p.o[head0 * 128 + idx] = 0;
        }
        return;
    }
    const int t0 = split * p.split_tokens;
    if (t0 >= L) return;                                     // uniform across the CTA
    if (pipeline_failed_before(p.err_count)) return;
    const int t1 = min(L, t0 + p.split_tokens);
    const int n_tiles = (t1 - t0 + kTile - 1) / kTile;
    const int n_splits = (L + p.split_tokens - 1) / p.split_tokens;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    __shared__ int timed_out;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        timed_out = 0;
        fence_mbarrier_init();
    }
    __syncthreads();

    const int32_t *bt = p.block_tables + (int64_t)b * p.max_blocks;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&k_map);
            tma_prefetch_desc(&v_map);
            for (int i = 0; i < n_tiles; ++i) {
                const int stage = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[stage], ((i / kStages) & 1) ^ 1)) {
                    timed_out = 1;
                    flag_pipeline_failure(p.err_count);
                    break;
                }
                const int tok = t0 + i * kTile;
                const int blk = __ldg(bt + tok / p.block_size);
                const int off = tok % p.block_size;
                if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                    count_error(p.err_count);
                    mbar_arrive(&full[stage]);          // consumers skip this tile
                    continue;
                }
                uint8_t *st = smem + stage * kStageBytes;
                mbar_arrive_expect_tx(&full[stage], kStageBytes);
                tma_load_4d(st, &k_map, &full[stage], 0, g, off, blk);
                tma_load_4d(st + kHalfTileBytes, &k_map, &full[stage], 64, g, off, blk);
                tma_load_4d(st + 2 * kHalfTileBytes, &v_map, &full[stage], 0, g, off, blk);
                tma_load_4d(st + 3 * kHalfTileBytes, &v_map, &full[stage], 64, g, off, blk);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int r = lane >> 2;          // accumulator row (query head) r and r + 8
    const int qd = lane & 3;          // column pair within an 8-wide n tile
    uint32_t qa[8][4];
    {
        const uint16_t *qrow0 = p.q + (int64_t)b * p.q_stride + (int64_t)(g * G + r) * 128;
        const uint16_t *qrow1 = qrow0 + 8 * 128;
        const bool v0 = r < G, v1 = r + 8 < G;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int c = kk * 16 + 2 * qd;
            qa[kk][0] = v0 ? __ldg(reinterpret_cast<const uint32_t *>(qrow0 + c)) : 0u;
            qa[kk][1] = v1 ? __ldg(reinterpret_cast<const uint32_t *>(qrow1 + c)) : 0u;
            qa[kk][2] = v0 ? __ldg(reinterpret_cast<const uint32_t *>(qrow0 + c + 8)) : 0u;
            qa[kk][3] = v1 ? __ldg(reinterpret_cast<const uint32_t *>(qrow1 + c + 8)) : 0u;
        }
    }
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = p.scale_log2;

    // ldmatrix lane roles: K (non-transposed) needs tokens (lane&7) + 8*(lane>>4)
    // and chunk offset (lane>>3)&1; V (transposed) needs tokens
    // (lane&7) + 8*((lane>>3)&1) and chunk offset lane>>4.
    const int k_tok = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
    const int k_chk = (lane >> 3) & 1;
    const int v_tok = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_chk = lane >> 4;

    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
        const int stage = i % kStages;
        if (!mbar_wait(&full[stage], (i / kStages) & 1)) {
            ok = false;
            if (lane == 0) flag_pipeline_failure(p.err_count);
            break;
        }
        const int tok0 = t0 + i * kTile + warp * 16;        // first token of this warp's slice
        int valid = t1 - tok0;
        valid = valid < 0 ? 0 : (valid > 16 ? 16 : valid);
        const int blk = __ldg(bt + (t0 + i * kTile) / p.block_size);
        if (blk < 0 || (int64_t)blk >= p.num_blocks) valid = 0;
        uint8_t *st = smem + stage * kStageBytes;
        const uint32_t kb = smem_u32(st), vb = smem_u32(st + 2 * kHalfTileBytes);
        if (valid > 0) {
            if (valid < 16) {
                // Keys past the context may hold any bits; their probability
                // is zero, but 0 * NaN is not, so clear those V rows.
                for (int e = lane; e < (16 - valid) * 16; e += 32) {
                    const int row = warp * 16 + valid + (e >> 4);
                    const int ch = e & 15;
                    uint8_t *hb = st + 2 * kHalfTileBytes + (ch >> 3) * kHalfTileBytes;
                    *reinterpret_cast<uint4 *>(hb + swz128(row, ch & 7)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S = Q K^T over this warp's 16 tokens (two n8 tiles)
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int ch = (kk & 3) * 2 + k_chk;
                const uint32_t addr = kb + (kk >> 2) * kHalfTileBytes + swz128(k_tok, ch);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(s[0], qa[kk], b0, b1);
                mma_bf16_16816(s[1], qa[kk], b2, b3);
            }
            // ---- mask, online softmax (base 2)
            float x[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = n * 8 + 2 * qd + (e & 1);
                    x[n][e] = col < valid ? s[n][e] * sl2 : -INFINITY;
                }
            float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            // valid > 0 makes mn finite; m may still be -inf on the first tile.
            const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float pr[2][4];
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                pr[n][0] = fast_exp2(x[n][0] - mn0);
                pr[n][1] = fast_exp2(x[n][1] - mn0);
                pr[n][2] = fast_exp2(x[n][2] - mn1);
                pr[n][3] = fast_exp2(x[n][3] - mn1);
                rs0 += pr[n][0] + pr[n][1];
                rs1 += pr[n][2] + pr[n][3];
            }
            l0 = l0 * a0 + rs0;
            l1 = l1 * a1 + rs1;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
            // ---- O += P V: P's accumulator layout is the A-operand layout
            const uint32_t pa[4] = {pack_bf16x2(pr[0][0], pr[0][1]), pack_bf16x2(pr[0][2], pr[0][3]),
                                    pack_bf16x2(pr[1][0], pr[1][1]), pack_bf16x2(pr[1][2], pr[1][3])};
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
                const int ch = c + v_chk;                   // 16-byte chunk of head_dim, 0..15
                const uint32_t addr = vb + (ch >> 3) * kHalfTileBytes + swz128(v_tok, ch & 7);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                mma_bf16_16816(o[c], pa, b0, b1);
                mma_bf16_16816(o[c + 1], pa, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // ---- combine the four warps (stage buffers are free once all consumers
    // are past their last tile: every TMA they waited on has landed and the
    // producer issues nothing after the last tile)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    named_barrier_consumers();
    float *comb_o = reinterpret_cast<float *>(smem);
    float *comb_m = comb_o + kConsumerWarps * 16 * kCombStride;
    float *comb_l = comb_m + kConsumerWarps * 16;
    if (!ok) timed_out = 1;
    {
        float *row0 = comb_o + (warp * 16 + r) * kCombStride;
        float *row1 = row0 + 8 * kCombStride;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            *reinterpret_cast<float2 *>(row0 + n * 8 + 2 * qd) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2 *>(row1 + n * 8 + 2 * qd) = make_float2(o[n][2], o[n][3]);
        }
        if (qd == 0) {
            comb_m[warp * 16 + r] = m0;
            comb_m[warp * 16 + r + 8] = m1;
            comb_l[warp * 16 + r] = l0;
            comb_l[warp * 16 + r + 8] = l1;
        }
    }
    named_barrier_consumers();
    // A wait that gave up leaves this split's keys unread: its result is
    // written as NaN, so neither the merge nor the caller can take it (or a
    // stale workspace slot) for an answer, even without an error counter.
    const bool failed = timed_out != 0;
    const int tid = threadIdx.x;                 // 0 .. 127
    for (int idx = tid; idx < G * 128; idx += kConsumerWarps * 32) {
        const int row = idx >> 7, d = idx & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb_m[w * 16 + row]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = comb_m[w * 16 + row];
            // A warp that saw no key (every tile of it skipped) adds nothing;
            // testing for it keeps -inf - -inf out of the exponent when no
            // warp of the split saw a key.
            const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
            num += f * comb_o[(w * 16 + row) * kCombStride + d];
            den += f * comb_l[w * 16 + row];
        }
        // den == 0 only if every key of the split was skipped (bad block
        // ids): the split then holds no key, its output is 0 and its
        // log-sum-exp -inf, so the merge gives it weight 0.
        float val = den > 0.f ? num / den : 0.f;
        float lse = den > 0.f ? M + log2f(den) : -INFINITY;
        if (failed) val = lse = __int_as_float(0x7fc00000);
        const int64_t head = head0 + row;
        if (n_splits == 1) {
            __nv_bfloat16 hv = __float2bfloat16_rn(val);
            p.o[head * 128 + d] = *reinterpret_cast<uint16_t *>(&hv);
        } else {
            const int64_t slot = head * p.max_splits + split;
            p.ws_o[slot * 128 + d] = val;
            if (d == 0) p.ws_lse[slot] = lse;
        }
    }
}

// One warp per (sequence, query head): combine the splits' partial outputs.
__global__ void __launch_bounds__(256)
decode_merge_kernel(const DecodeParams p) {
    pdl_wait_release();
    const int64_t wid = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const bool valid = wid < (int64_t)p.B * p.Hq;
    // The context length is requested before the failure flag is read, so
    // the two round trips overlap.
    int L = valid ? __ldg(p.context_lens + wid / p.Hq) : 0;
    // After a pipeline failure (this call's or an earlier one's, bit 30 of
    // err_count) some splits wrote nothing: their workspace slots may hold an
    // earlier call's partials.  Merge nothing and leave o as it is, as the
    // split kernel does for the sequences it did not process.
    if (pipeline_failed_before(p.err_count)) return;
    if (!valid) return;
    const int max_l = p.max_blocks * p.block_size;
    L = L < 0 ? 0 : (L > max_l ? max_l : L);
    const int n_splits = (L + p.split_tokens - 1) / p.split_tokens;
    if (n_splits <= 1) return;                  // written by the split kernel
    const float *lse = p.ws_lse + wid * p.max_splits;
    const float4 *part = reinterpret_cast<const float4 *>(p.ws_o + wid * p.max_splits * 128) + lane;
    float M = -INFINITY;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
    // A split whose keys were all skipped has lse = -inf and weight 0.
    auto add = [&](float ls, float4 v) {
        const float f = ls == -INFINITY ? 0.f : fast_exp2(ls - M);
        acc[0] = fmaf(f, v.x, acc[0]);
        acc[1] = fmaf(f, v.y, acc[1]);
        acc[2] = fmaf(f, v.z, acc[2]);
        acc[3] = fmaf(f, v.w, acc[3]);
        den += f;
    };
    constexpr int kInFlight = 8;
    if (n_splits <= kInFlight) {
        // Every load of the merge in one round trip.
        float ls[kInFlight];
        float4 v[kInFlight];
#pragma unroll
        for (int s = 0; s < kInFlight; ++s) {
            ls[s] = s < n_splits ? lse[s] : -INFINITY;
            v[s] = s < n_splits ? part[s * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int s = 0; s < kInFlight; ++s) M = fmaxf(M, ls[s]);
        if (M != -INFINITY) {
#pragma unroll
            for (int s = 0; s < kInFlight; ++s) add(ls[s], v[s]);
        }
    } else {
        for (int s = 0; s < n_splits; ++s) M = fmaxf(M, lse[s]);
        if (M != -INFINITY)
            for (int s = 0; s < n_splits; ++s) add(lse[s], part[s * 32]);
    }
    uint2 out = make_uint2(0u, 0u);             // every key of the sequence skipped
    if (M != -INFINITY) {
        const float inv = 1.f / den;
        out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    }
    *reinterpret_cast<uint2 *>(p.o + wid * 128 + 4 * lane) = out;
}

int decode_resolve_split(int B, int Hkv, int max_blocks, int block_size, int kv_split_tokens,
                         int num_sms) {
    const int64_t max_ctx = (int64_t)max_blocks * block_size;
    const int64_t cap = (max_ctx + kTile - 1) / kTile * kTile;
    int64_t split;
    if (kv_split_tokens > 0) {
        split = (kv_split_tokens + kTile - 1) / kTile * kTile;
    } else {
        // Each split pays a fixed cost (pipeline fill, its partial result and
        // its share of the merge), so long splits win while the grid still
        // balances: the longest of 4096 .. 1536 keys that leaves the longest
        // context at least four splits and the grid twelve CTAs per SM.
        // (Measured on GB300 against fixed splits: the best or within 1% on
        // B = 64 x 4k, 256 x 8k and 32 x 40k contexts; 1024-key splits lost
        // 5% on the last.)
        //
        // Otherwise (short contexts, or few sequences for their length):
        // 1024 keys, or no split at all when the longest context is at most
        // 2048 keys and there are at least as many (sequence, kv head) pairs
        // as SMs; halved (to >= 512) only while the grid has fewer CTAs than
        // half the SMs.  Here the fixed cost of a CTA (first loads, combine,
        // partial result) and of the merge outweighs spreading the keys:
        // sweeps over B = 8..256 with contexts up to 8192 keys, uniform and
        // varied, found 256- and 512-key splits slower than 1024 almost
        // everywhere (by up to 30%, at B = 16..64 with contexts of 512 to
        // 2048 keys), even where the longer splits leave the grid below one
        // CTA per SM.
        //
        // A single long sequence, too short of CTAs for that, takes the
        // longest of those splits that fills the GPU in one wave of one or
        // two CTAs per SM (40960 keys: 2048-key splits, 26% faster than
        // 1024).  With two or more sequences the host sees only the longest
        // context: shorter ones leave such a grid half empty (B = 2, 4 with
        // contexts up to 40960 keys ran 15-30% slower so), and the rule
        // below applies.
        const int64_t pairs = (int64_t)B * Hkv;
        split = 0;
        for (const int64_t cand : {4096, 3072, 2048, 1536}) {
            const int64_t ctas = pairs * ((max_ctx + cand - 1) / cand);
            if (4 * cand <= max_ctx &&
                (ctas >= 12LL * num_sms ||
                 (B == 1 && ctas >= num_sms && ctas <= 2LL * num_sms))) {
                split = cand;
                break;
            }
        }
        if (split == 0) {
            split = (max_ctx <= 2048 && pairs >= num_sms) ? 2048 : 1024;
            while (split > 512 && 2 * pairs * ((max_ctx + split - 1) / split) < num_sms)
                split /= 2;
        }
    }
    if (split > cap) split = cap;
    if (split < kTile) split = kTile;
    return (int)split;
}

size_t decode_workspace_bytes(int B, int Hq, int max_splits) {
    if (max_splits <= 1) return 0;
    const size_t n = (size_t)B * Hq * max_splits;
    return n * 128 * sizeof(float) + n * sizeof(float);
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, cudaStream_t s) {
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = ensure_dynamic_smem(decode_split_kernel, kDecodeSmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    if (p.B == 0) return cudaSuccess;
    dim3 grid(p.max_splits, p.Hkv, p.B);
    e = launch_pdl(decode_split_kernel, grid, dim3(kDecodeThreads), (size_t)kDecodeSmemBytes, s,
                   k_map, v_map, p);
    if (e == cudaErrorInvalidValue || e == cudaErrorInvalidConfiguration) {
        // The shared-memory attribute was lost (the device was reset): set it again, retry once.
        cudaGetLastError();
        e = ensure_dynamic_smem(decode_split_kernel, kDecodeSmemBytes, smem_set, true);
        if (e == cudaSuccess)
            e = launch_pdl(decode_split_kernel, grid, dim3(kDecodeThreads),
                           (size_t)kDecodeSmemBytes, s, k_map, v_map, p);
    }
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    const int64_t warps = (int64_t)p.B * p.Hq;
    return launch_pdl(decode_merge_kernel, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256),
                      (size_t)0, s, p);
}

}  // namespace nvattn
