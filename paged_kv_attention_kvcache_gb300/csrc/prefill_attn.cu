// Varlen causal prefill attention on tcgen05 tensor cores.
//
// What it computes ("3.3 Model skeleton and core operators", sec. 7.2;
// "同一个 Qwen3，两种写法", sec. 3.2; "Nano-vLLM 源码解读 第17篇", sec. 5.2): for
// each packed sequence, query head h and query row i,
// o_i = sum_{j <= i} softmax_j(scale * q_i . k_j) v_j with k, v from kv head
// h / (Hq / Hkv).  The mask is block-diagonal over sequences and causal
// inside each; keys of other sequences are never admitted.
//
// How (GB300):
//  - One CTA per (128-row query tile, query head, sequence).  The grid's z
//    index runs over query tiles from the last (most keys under the causal
//    mask) to the first, so the heaviest CTAs are dispatched first.
//  - Warp 4 issues TMA loads: the Q tile once, then 128-token K and V tiles
//    into two-deep rings (K and V have separate barriers so QK^T can start
//    before V lands).  Every tile is stored as two 128-byte-swizzled halves
//    of head_dim, the canonical layout tcgen05 reads.
//  - Warp 5 allocates tensor memory (512 columns: two S buffers and O) and one
//    of its threads issues tcgen05.mma: S_j = Q K_j^T (M=N=128, K=128, bf16
//    in, fp32 accumulate in TMEM), then O += P_{j-1} V_{j-1} with P from
//    shared memory (K-major) and V read MN-major.  S_{j+1} overlaps the
//    softmax of S_j.
//  - Warps 0-3 own one query row per thread (TMEM lane = row): tcgen05.ld of
//    the S row, causal mask on the diagonal tile, online softmax in base 2
//    with a lazy rescale (O in TMEM is rescaled only when the running max
//    grows by more than 2^8, so the stale max bounds p by 256), P written as
//    bf16 into swizzled shared memory, and finally O / l to global memory.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace nvattn {

namespace {

constexpr int kBM = 128;                        // query rows per CTA
constexpr int kBN = 128;                        // keys per KV tile
constexpr int kHalf = 128 * 128;                // 128 rows x 64 dims x 2 B = 16 KB
constexpr int kTileBytes = 2 * kHalf;           // one Q / K / V / P tile, 32 KB
constexpr int kKVStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kKVStages * kTileBytes;
constexpr int kOffP = kOffV + kKVStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
constexpr int kPrefillThreads = 192;            // 4 softmax warps, TMA warp, MMA warp
constexpr int kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: rescale when max grows > 2^8

struct Barriers {
    uint64_t q_full;
    uint64_t k_full[kKVStages], v_full[kKVStages];
    uint64_t k_empty[kKVStages], v_empty[kKVStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, pv_done;
    uint32_t tmem_base;
    int failed;
};
constexpr int kPrefillSmemBytes = kOffBar + (int)sizeof(Barriers) + 1024;

// ------------------------------------------------------------ tcgen05 PTX
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, tcgen05 version bits.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
          "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
          "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void record_failure(Barriers *bars, int *err_count) {
    if (atomicExch(&bars->failed, 1) == 0) flag_pipeline_failure(err_count);
}

}  // namespace

__global__ void __launch_bounds__(kPrefillThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const PrefillParams p) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int qt = (int)gridDim.z - 1 - (int)blockIdx.z;   // heaviest tiles first
    const int q_start = __ldg(p.cu_seqlens_q + b);
    const int L = __ldg(p.cu_seqlens_q + b + 1) - q_start;
    const int k_start = __ldg(p.cu_seqlens_k + b);
    const int q0 = qt * kBM;
    if (q0 >= L) return;                                    // uniform across the CTA
    if (pipeline_failed_before(p.err_count)) return;
    const int n_kv = qt + 1;                                 // causal: key tiles 0..qt
    const int kvh = h / (p.Hq / p.Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers *bars = reinterpret_cast<Barriers *>(smem + kOffBar);

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < kKVStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->s_free[s], 4);
        }
        mbar_init(&bars->p_full, 4);
        mbar_init(&bars->pv_done, 1);
        bars->failed = 0;
        fence_mbarrier_init();
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&bars->tmem_base)), "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    uint8_t *sQ = smem + kOffQ;
    uint8_t *sP = smem + kOffP;

    if (warp == 4) {
        // ------------------------------------------------------------- TMA
        if (lane == 0) {
            tma_prefetch_desc(&q_map);
            tma_prefetch_desc(&k_map);
            tma_prefetch_desc(&v_map);
            mbar_arrive_expect_tx(&bars->q_full, kTileBytes);
            tma_load_3d(sQ, &q_map, &bars->q_full, 0, h, q_start + q0);
            tma_load_3d(sQ + kHalf, &q_map, &bars->q_full, 64, h, q_start + q0);
            for (int j = 0; j < n_kv; ++j) {
                const int st = j & 1;
                const uint32_t par = ((j >> 1) - 1) & 1;
                const int row = k_start + j * kBN;
                uint8_t *sK = smem + kOffK + st * kTileBytes;
                uint8_t *sV = smem + kOffV + st * kTileBytes;
                if (j >= kKVStages && !mbar_wait(&bars->k_empty[st], par)) {
                    record_failure(bars, p.err_count);
                    break;
                }
                mbar_arrive_expect_tx(&bars->k_full[st], kTileBytes);
                tma_load_3d(sK, &k_map, &bars->k_full[st], 0, kvh, row);
                tma_load_3d(sK + kHalf, &k_map, &bars->k_full[st], 64, kvh, row);
                if (j >= kKVStages && !mbar_wait(&bars->v_empty[st], par)) {
                    record_failure(bars, p.err_count);
                    break;
                }
                mbar_arrive_expect_tx(&bars->v_full[st], kTileBytes);
                tma_load_3d(sV, &v_map, &bars->v_full[st], 0, kvh, row);
                tma_load_3d(sV + kHalf, &v_map, &bars->v_full[st], 64, kvh, row);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_bf16(kBM, kBN, false);
            constexpr uint32_t kIdescPV = idesc_bf16(kBM, 128, true);
            const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
            bool ok = mbar_wait(&bars->q_full, 0);
            for (int j = 0; ok && j <= n_kv; ++j) {
                if (j < n_kv) {
                    const int st = j & 1, sb = j & 1;
                    if (!mbar_wait(&bars->k_full[st], (j >> 1) & 1) ||
                        (j >= 2 && !mbar_wait(&bars->s_free[sb], ((j >> 1) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(smem + kOffK + st * kTileBytes);
                    const uint32_t d = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
                        tc_mma(d, smem_desc_sw128(q_addr + off, 16, 1024),
                               smem_desc_sw128(k_addr + off, 16, 1024), kIdescQK, kk > 0);
                    }
                    tc_commit(&bars->s_full[sb]);
                    tc_commit(&bars->k_empty[st]);
                }
                if (j >= 1) {
                    const int jj = j - 1, st = jj & 1;
                    if (!mbar_wait(&bars->p_full, jj & 1) ||
                        !mbar_wait(&bars->v_full[st], (jj >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t v_addr = smem_u32(smem + kOffV + st * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // P: K-major like Q.  V: MN-major; 16 keys = 2 swizzle atoms
                        // (2048 B) per step, the second 64 dims 16 KB (LBO) away.
                        const uint32_t poff = (kk >> 2) * kHalf + (kk & 3) * 32;
                        tc_mma(tmem + kColO, smem_desc_sw128(p_addr + poff, 16, 1024),
                               smem_desc_sw128(v_addr + kk * 2048, kHalf, 1024), kIdescPV,
                               (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&bars->pv_done);
                    tc_commit(&bars->v_empty[st]);
                }
            }
            if (!ok) record_failure(bars, p.err_count);
        }
    } else {
        // --------------------------------------------------------- softmax
        const int row = warp * 32 + lane;                 // TMEM lane = query row in tile
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            if (!mbar_wait(&bars->s_full[sb], (j >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_addr + (sb ? kColS1 : kColS0) + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[sb]);
            if (j == n_kv - 1) {
                // Diagonal tile (query and key tiles both start at q0): key c
                // is visible to row `row` iff c <= row.
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > row) s[c] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
            const float m_new = fmaxf(m_used, mx * sl2);
            float alpha = 1.f;
            const bool rescale = m_new > m_used + kRescaleThreshold;
            if (rescale) {
                alpha = fast_exp2(m_used - m_new);      // 0 on the first tile
                m_used = m_new;
            }
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float p0 = fast_exp2(fmaf(s[2 * c], sl2, -m_used));
                const float p1 = fast_exp2(fmaf(s[2 * c + 1], sl2, -m_used));
                sum += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l = fmaf(l, alpha, sum);
            if (j >= 1) {
                // O and the P buffer are busy until PV_{j-1} completes.
                if (!mbar_wait(&bars->pv_done, (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(lane_addr + kColO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st32(lane_addr + kColO + c * 32, r);
                    }
                    tmem_wait_st();
                }
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint8_t *dst = sP + (c >> 3) * kHalf + swz128(row, c & 7);
                *reinterpret_cast<uint4 *>(dst) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);
        }
        if (ok && mbar_wait(&bars->pv_done, (n_kv - 1) & 1)) {
            tc_fence_after();
            const int qpos = q0 + row;
            const float inv_l = 1.f / l;
            uint16_t *orow = p.o + ((int64_t)(q_start + qpos) * p.Hq + h) * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_addr + kColO + c * 32, r);
                tmem_wait_ld();
                if (qpos < L) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(r[8 * e]) * inv_l, __uint_as_float(r[8 * e + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * inv_l, __uint_as_float(r[8 * e + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * inv_l, __uint_as_float(r[8 * e + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * inv_l, __uint_as_float(r[8 * e + 7]) * inv_l);
                        *reinterpret_cast<uint4 *>(orow + c * 32 + 8 * e) = v;
                    }
                }
            }
        } else {
            record_failure(bars, p.err_count);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(kTmemCols));
    }
}

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map,
                           cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kPrefillSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int n_qt = (p.max_seqlen_q + kBM - 1) / kBM;
    if (p.B == 0 || n_qt == 0) return cudaSuccess;
    dim3 grid(p.Hq, p.B, n_qt);
    prefill_attn_kernel<<<grid, kPrefillThreads, kPrefillSmemBytes, s>>>(q_map, k_map, v_map, p);
    return cudaGetLastError();
}

}  // namespace nvattn
