// Elementwise / row-reduction kernels of the attention sublayer: the RoPE
// table, fused residual-add RMSNorm and per-head QK-Norm + RoPE.  All are
// HBM-bound; they move 16-byte vectors, keep the row in registers, reduce
// with warp shuffles and compute in fp32.
#include "common.cuh"
#include "internal.h"

namespace nvattn {

// ------------------------------------------------------------- RoPE table
// "3.3 Model skeleton and core operators", sec. 3: row p holds
// cos(p * inv_freq[i]) for i < half, then sin(p * inv_freq[i]).  The angle is
// formed in fp64 so that only the final value is rounded to fp32.
__global__ void rope_cos_sin_kernel(float *__restrict__ cos_sin, int max_position,
                                    int rotary_dim, double base) {
    pdl_wait_release();
    const int half = rotary_dim / 2;
    const int64_t n = (int64_t)max_position * half;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = idx / half;
        const int i = (int)(idx % half);
        const double inv_freq = 1.0 / pow(base, (double)(2 * i) / (double)rotary_dim);
        const double angle = (double)p * inv_freq;
        double sv, cv;
        sincos(angle, &sv, &cv);
        cos_sin[p * rotary_dim + i] = (float)cv;
        cos_sin[p * rotary_dim + half + i] = (float)sv;
    }
}

cudaError_t launch_rope_cos_sin(float *cos_sin, int max_position, int rotary_dim, double base,
                                cudaStream_t s) {
    const int64_t n = (int64_t)max_position * (rotary_dim / 2);
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(rope_cos_sin_kernel, dim3((unsigned)blocks), dim3(threads), (size_t)0, s,
                      cos_sin, max_position, rotary_dim, base);
}

// --------------------------------------------------------- add + RMSNorm
// "3.3 Model skeleton and core operators", sec. 2 and "同一个 Qwen3，两种写法",
// sec. 3.6: one CTA per row; each thread owns VPT 16-byte vectors (8 bf16) of
// the row, so the row is read once, the fp32 sum stays in registers, and the
// row is written twice (residual_out, out): 32 KiB per token at H = 4096.
constexpr int kNormThreads = 128;

template <int VPT, bool kResidual>
__global__ void __launch_bounds__(kNormThreads)
add_rmsnorm_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ residual,
                   const uint4 *__restrict__ weight, uint4 *__restrict__ out,
                   uint4 *__restrict__ residual_out, int nvec, int64_t vstride, float inv_h,
                   float eps) {
    pdl_wait_release();
    const int64_t row = blockIdx.x;
    const int64_t row0 = row * vstride;          // first 16-byte vector of the row
    const uint4 *xr = x + row0;
    float s[VPT][8];
    float sum_sq = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = threadIdx.x + v * kNormThreads;
        if (c < nvec) {
            uint4 a = __ldg(xr + c);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[v][2 * e] = bf16_lo(aw[e]);
                s[v][2 * e + 1] = bf16_hi(aw[e]);
            }
            if (kResidual) {
                uint4 r = __ldg(residual + row0 + c);
                const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s[v][2 * e] += bf16_lo(rw[e]);
                    s[v][2 * e + 1] += bf16_hi(rw[e]);
                    o[e] = pack_bf16x2(s[v][2 * e], s[v][2 * e + 1]);
                }
                residual_out[row0 + c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sum_sq = fmaf(s[v][e], s[v][e], sum_sq);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum_sq += __shfl_xor_sync(0xffffffffu, sum_sq, off);
    __shared__ float warp_sums[kNormThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = sum_sq;
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) total += warp_sums[w];
    const float rstd = rsqrtf(total * inv_h + eps);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = threadIdx.x + v * kNormThreads;
        if (c < nvec) {
            uint4 g = __ldg(weight + c);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack_bf16x2(s[v][2 * e] * rstd * bf16_lo(gw[e]),
                                   s[v][2 * e + 1] * rstd * bf16_hi(gw[e]));
            out[row0 + c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

template <int VPT>
static cudaError_t launch_norm_vpt(const uint16_t *x, const uint16_t *residual,
                                   const uint16_t *weight, uint16_t *out,
                                   uint16_t *residual_out, int64_t T, int H,
                                   int64_t row_stride, float eps, cudaStream_t s) {
    const int nvec = H / 8;
    const int64_t vstride = row_stride / 8;
    const float inv_h = 1.0f / (float)H;
    dim3 grid((unsigned)T);
    if (residual)
        return launch_pdl(add_rmsnorm_kernel<VPT, true>, grid, dim3(kNormThreads), (size_t)0, s,
                          (const uint4 *)x, (const uint4 *)residual, (const uint4 *)weight,
                          (uint4 *)out, (uint4 *)residual_out, nvec, vstride, inv_h, eps);
    return launch_pdl(add_rmsnorm_kernel<VPT, false>, grid, dim3(kNormThreads), (size_t)0, s,
                      (const uint4 *)x, (const uint4 *)nullptr, (const uint4 *)weight,
                      (uint4 *)out, (uint4 *)nullptr, nvec, vstride, inv_h, eps);
}

cudaError_t launch_add_rmsnorm(const uint16_t *x, const uint16_t *residual,
                               const uint16_t *weight, uint16_t *out, uint16_t *residual_out,
                               int64_t T, int H, int64_t row_stride, float eps, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int nvec = H / 8;
    const int vpt = (nvec + kNormThreads - 1) / kNormThreads;
#define NV_NORM_ARGS x, residual, weight, out, residual_out, T, H, row_stride, eps, s
    if (vpt <= 1) return launch_norm_vpt<1>(NV_NORM_ARGS);
    if (vpt <= 2) return launch_norm_vpt<2>(NV_NORM_ARGS);
    if (vpt <= 4) return launch_norm_vpt<4>(NV_NORM_ARGS);
    if (vpt <= 8) return launch_norm_vpt<8>(NV_NORM_ARGS);
    return launch_norm_vpt<16>(NV_NORM_ARGS);
#undef NV_NORM_ARGS
}

// ------------------------------------------------------- QK-Norm + RoPE
// "3.3 Model skeleton and core operators", sec. 8 and sec. 3: for each
// (token, head) row of 128 elements, RMSNorm over the row with the q_norm or
// k_norm weight, then rotate the pair (i, i + 64) by the position's angle.
// Eight lanes own one row: lane j holds elements [8j, 8j+8) of the first half
// and [64 + 8j, 64 + 8j + 8) of the second, so each lane has both members of
// its eight pairs and the rotation needs no exchange.  Four rows per warp.
constexpr int kRopeThreads = 256;

// Normalise and rotate one 128-element head row.  The eight lanes of the
// group named by `gmask` each hold elements [8j, 8j+8) (in a) and
// [64+8j, 64+8j+8) (in b) of the row; on return out1/out2 hold the lane's
// rotated elements as packed bf16 pairs.  Shared by the in-place kernel and
// the fused cache-writing one so that both give the same bits.
__device__ __forceinline__ void norm_rope_regs(uint4 a, uint4 b, const uint16_t *__restrict__ w,
                                               const float *__restrict__ cs_row, int j,
                                               unsigned gmask, float eps, uint4 &out1,
                                               uint4 &out2) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    float x1[8], x2[8];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x1[2 * e] = bf16_lo(aw[e]);
        x1[2 * e + 1] = bf16_hi(aw[e]);
        x2[2 * e] = bf16_lo(bw[e]);
        x2[2 * e + 1] = bf16_hi(bw[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(x1[e], x1[e], fmaf(x2[e], x2[e], ss));
    ss += __shfl_xor_sync(gmask, ss, 4);
    ss += __shfl_xor_sync(gmask, ss, 2);
    ss += __shfl_xor_sync(gmask, ss, 1);
    const float rstd = rsqrtf(ss * (1.0f / 128.0f) + eps);
    const uint4 wa = __ldg(reinterpret_cast<const uint4 *>(w + 8 * j));
    const uint4 wb = __ldg(reinterpret_cast<const uint4 *>(w + 64 + 8 * j));
    const uint32_t waw[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wbw[4] = {wb.x, wb.y, wb.z, wb.w};
    const float4 *cs = reinterpret_cast<const float4 *>(cs_row);
    const float4 c0 = __ldg(cs + 2 * j), c1 = __ldg(cs + 2 * j + 1);
    const float4 s0 = __ldg(cs + 16 + 2 * j), s1 = __ldg(cs + 16 + 2 * j + 1);
    const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float n1[2], n2[2];
        n1[0] = x1[2 * e] * rstd * bf16_lo(waw[e]);
        n1[1] = x1[2 * e + 1] * rstd * bf16_hi(waw[e]);
        n2[0] = x2[2 * e] * rstd * bf16_lo(wbw[e]);
        n2[1] = x2[2 * e + 1] * rstd * bf16_hi(wbw[e]);
        float y1[2], y2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float c = cv[2 * e + u], sn = sv[2 * e + u];
            y1[u] = n1[u] * c - n2[u] * sn;
            y2[u] = n2[u] * c + n1[u] * sn;
        }
        o1[e] = pack_bf16x2(y1[0], y1[1]);
        o2[e] = pack_bf16x2(y2[0], y2[1]);
    }
    out1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    out2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

// The same, loading the lane's two vectors from `src` first.
__device__ __forceinline__ void norm_rope_row(const uint16_t *src, const uint16_t *__restrict__ w,
                                              const float *__restrict__ cs_row, int j,
                                              unsigned gmask, float eps, uint4 &out1,
                                              uint4 &out2) {
    const uint4 a = *reinterpret_cast<const uint4 *>(src + 8 * j);
    const uint4 b = *reinterpret_cast<const uint4 *>(src + 64 + 8 * j);
    norm_rope_regs(a, b, w, cs_row, j, gmask, eps, out1, out2);
}

// Each 8-lane group walks rows row0, row0 + groups, ... and loads the next
// row's vectors and position before it normalises and rotates the current
// one, so the SM always has loads in flight instead of running one dependent
// load -> table -> compute chain per row and exiting.
__global__ void __launch_bounds__(kRopeThreads)
qknorm_rope_kernel(uint16_t *__restrict__ q, int64_t q_stride, uint16_t *__restrict__ k,
                   int64_t k_stride, const uint16_t *__restrict__ qw,
                   const uint16_t *__restrict__ kw, const float *__restrict__ cos_sin,
                   int max_position, const int64_t *__restrict__ positions, int64_t T, int Hq,
                   int Hkv, float eps, int *err_count) {
    pdl_wait_release();
    const int heads = Hq + Hkv;
    const int64_t n_rows = T * heads;
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;                       // lane within the row group
    const int64_t groups = (int64_t)gridDim.x * (kRopeThreads / 8);
    int64_t row = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 3;
    if (row >= n_rows) return;
    // Groups of the same warp may leave the loop at different rows, so the
    // row's shuffles name only this group's lanes; all eight share the row.
    const unsigned gmask = 0xFFu << (lane & ~7);
    auto locate = [&](int64_t r, int64_t &t) {
        t = r / heads;
        const int h = (int)(r - t * heads);
        return h < Hq ? q + t * q_stride + (int64_t)h * 128
                      : k + t * k_stride + (int64_t)(h - Hq) * 128;
    };
    int64_t t;
    uint16_t *base = locate(row, t);
    const uint16_t *w = (row % heads) < Hq ? qw : kw;
    uint4 a = *reinterpret_cast<const uint4 *>(base + 8 * j);
    uint4 b = *reinterpret_cast<const uint4 *>(base + 64 + 8 * j);
    int64_t pos = __ldg(positions + t);
    for (;;) {
        const int64_t next = row + groups;
        const bool more = next < n_rows;
        uint16_t *nbase = base;
        int64_t nt = t;
        uint4 na = a, nb = b;
        int64_t npos = pos;
        if (more) {
            nbase = locate(next, nt);
            na = *reinterpret_cast<const uint4 *>(nbase + 8 * j);
            nb = *reinterpret_cast<const uint4 *>(nbase + 64 + 8 * j);
            npos = __ldg(positions + nt);
        }
        if (pos < 0 || pos >= max_position) {
            if (j == 0) count_error(err_count);
        } else {
            uint4 o1, o2;
            norm_rope_regs(a, b, w, cos_sin + pos * 128, j, gmask, eps, o1, o2);
            *reinterpret_cast<uint4 *>(base + 8 * j) = o1;
            *reinterpret_cast<uint4 *>(base + 64 + 8 * j) = o2;
        }
        if (!more) break;
        w = (next % heads) < Hq ? qw : kw;
        row = next;
        base = nbase;
        t = nt;
        a = na;
        b = nb;
        pos = npos;
    }
}

cudaError_t launch_qknorm_rope(uint16_t *q, int64_t q_stride, uint16_t *k, int64_t k_stride,
                               const uint16_t *qw, const uint16_t *kw, const float *cos_sin,
                               int max_position, const int64_t *positions, int64_t T, int Hq,
                               int Hkv, float eps, int *err_count, cudaStream_t s) {
    const int64_t rows = T * (Hq + Hkv);
    if (rows == 0) return cudaSuccess;
    const int64_t threads = rows * 8;
    static const int64_t resident = resident_grid(qknorm_rope_kernel, kRopeThreads, 4);
    int64_t blocks = (threads + kRopeThreads - 1) / kRopeThreads;
    if (blocks > resident) blocks = resident;
    return launch_pdl(qknorm_rope_kernel, dim3(blocks), dim3(kRopeThreads), (size_t)0, s, q,
                      q_stride, k, k_stride, qw, kw, cos_sin, max_position, positions, T, Hq, Hkv,
                      eps, err_count);
}

// ------------------------------------------ QK-Norm + RoPE + store_kvcache
// The same per-row arithmetic as qknorm_rope_kernel, with the cache scatter of
// store_kvcache folded in ("Nano-vLLM 源码解读 第17篇", sec. 4 and 5.1 give
// the order: rotate q and k, then write k and v to their slots).  A token owns
// Hq + 2 Hkv rows of 128 elements: q rows are rotated in place, k rows are
// rotated and written to the token's cache slot (and back in place only when
// asked), v rows are copied bit for bit to the slot.  k never makes the extra
// round trip through HBM that the separate store kernel would read it back
// for.  Two phases, each with the grid's stride:
//  - the q and k rows, eight lanes per row as above;
//  - the v rows, one warp per token, all of the token's 16-byte loads issued
//    before its stores (the copy pattern of store_kvcache_kernel, which keeps
//    more bytes in flight than the rotation's row groups do).
// Four blocks per SM (64 registers, a few bytes spilled) measured faster
// than three without the spill: the loads in flight per SM are what count.
constexpr int kVCopyMaxVecPerLane = 8;    // D <= 2048 in one pass

__global__ void __launch_bounds__(kRopeThreads, 4)
qknorm_rope_store_kernel(uint16_t *__restrict__ q, int64_t q_stride, uint16_t *__restrict__ k,
                         int64_t k_stride, const uint16_t *__restrict__ v, int64_t v_stride,
                         const uint16_t *__restrict__ qw, const uint16_t *__restrict__ kw,
                         const float *__restrict__ cos_sin, int max_position,
                         const int64_t *__restrict__ positions,
                         const int32_t *__restrict__ slot_mapping, uint16_t *__restrict__ k_cache,
                         uint16_t *__restrict__ v_cache, int64_t num_slots, int64_t T, int Hq,
                         int Hkv, float eps, int write_k, int *err_count) {
    pdl_wait_release();
    const int heads = Hq + Hkv;                   // rows of the rotation phase per token
    const int64_t n_rows = T * heads;
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;
    const int64_t groups = (int64_t)gridDim.x * (kRopeThreads / 8);
    const int64_t D = (int64_t)Hkv * 128;
    const unsigned gmask = 0xFFu << (lane & ~7);
    // ---- phase 1: q and k rows.  Grid-stride over rows as in
    // qknorm_rope_kernel: the next row's vectors, position and slot are in
    // flight while the current row is processed.
    int64_t row = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 3;
    if (row < n_rows) {
        auto source = [&](int64_t t, int h) -> uint16_t * {
            return h < Hq ? q + t * q_stride + (int64_t)h * 128
                          : k + t * k_stride + (int64_t)(h - Hq) * 128;
        };
        int64_t t = row / heads;
        int h = (int)(row - t * heads);
        uint16_t *base = source(t, h);
        uint4 a = *reinterpret_cast<const uint4 *>(base + 8 * j);
        uint4 b = *reinterpret_cast<const uint4 *>(base + 64 + 8 * j);
        int64_t pos = __ldg(positions + t);
        int64_t slot = h >= Hq ? (int64_t)__ldg(slot_mapping + t) : -1;
        for (;;) {
            const int64_t next = row + groups;
            const bool more = next < n_rows;
            int64_t nt = t, npos = pos, nslot = slot;
            int nh = h;
            uint16_t *nbase = base;
            uint4 na = a, nb = b;
            if (more) {
                nt = next / heads;
                nh = (int)(next - nt * heads);
                nbase = source(nt, nh);
                na = *reinterpret_cast<const uint4 *>(nbase + 8 * j);
                nb = *reinterpret_cast<const uint4 *>(nbase + 64 + 8 * j);
                npos = __ldg(positions + nt);
                nslot = nh >= Hq ? (int64_t)__ldg(slot_mapping + nt) : -1;
            }
            if (slot != -1 && (slot < 0 || slot >= num_slots)) {
                if (j == 0 && h == Hq) count_error(err_count);   // once per token
                slot = -1;
            }
            if (pos < 0 || pos >= max_position) {
                if (j == 0) count_error(err_count);
            } else {
                const bool is_q = h < Hq;
                uint4 o1, o2;
                norm_rope_regs(a, b, is_q ? qw : kw, cos_sin + pos * 128, j, gmask, eps, o1, o2);
                if (is_q || write_k) {
                    *reinterpret_cast<uint4 *>(base + 8 * j) = o1;
                    *reinterpret_cast<uint4 *>(base + 64 + 8 * j) = o2;
                }
                if (!is_q && slot >= 0) {
                    uint16_t *dst = k_cache + slot * D + (int64_t)(h - Hq) * 128;
                    *reinterpret_cast<uint4 *>(dst + 8 * j) = o1;
                    *reinterpret_cast<uint4 *>(dst + 64 + 8 * j) = o2;
                }
            }
            if (!more) break;
            row = next;
            t = nt;
            h = nh;
            base = nbase;
            a = na;
            b = nb;
            pos = npos;
            slot = nslot;
        }
    }
    // ---- phase 2: v rows, a bit copy (a bad slot was counted in phase 1).
    const int vec = (int)(D / 8);
    const int64_t warps = (int64_t)gridDim.x * (kRopeThreads / 32);
    const uint4 *vv = reinterpret_cast<const uint4 *>(v);
    uint4 *vc = reinterpret_cast<uint4 *>(v_cache);
    for (int64_t t = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5; t < T; t += warps) {
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0 || slot >= num_slots) continue;
        const uint4 *src = vv + t * (v_stride / 8);
        for (int c0 = 0; c0 < vec; c0 += 32 * kVCopyMaxVecPerLane) {
            uint4 x[kVCopyMaxVecPerLane];
#pragma unroll
            for (int u = 0; u < kVCopyMaxVecPerLane; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < vec) x[u] = __ldg(src + c);
            }
#pragma unroll
            for (int u = 0; u < kVCopyMaxVecPerLane; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < vec) vc[slot * vec + c] = x[u];
            }
        }
    }
}

cudaError_t launch_qknorm_rope_store(uint16_t *q, int64_t q_stride, uint16_t *k,
                                     int64_t k_stride, const uint16_t *v, int64_t v_stride,
                                     const uint16_t *qw, const uint16_t *kw,
                                     const float *cos_sin, int max_position,
                                     const int64_t *positions, const int32_t *slot_mapping,
                                     uint16_t *k_cache, uint16_t *v_cache, int64_t num_slots,
                                     int64_t T, int Hq, int Hkv, float eps, int write_k,
                                     int *err_count, cudaStream_t s) {
    const int64_t rows = T * (Hq + Hkv);
    if (rows == 0) return cudaSuccess;
    const int64_t threads = rows * 8;
    static const int64_t resident = resident_grid(qknorm_rope_store_kernel, kRopeThreads, 4);
    int64_t blocks = (threads + kRopeThreads - 1) / kRopeThreads;
    if (blocks > resident) blocks = resident;
    return launch_pdl(qknorm_rope_store_kernel, dim3(blocks), dim3(kRopeThreads), (size_t)0, s, q,
                      q_stride, k, k_stride, v, v_stride, qw, kw, cos_sin, max_position,
                      positions, slot_mapping, k_cache, v_cache, num_slots, T, Hq, Hkv, eps,
                      write_k, err_count);
}

}  // namespace nvattn
