// combine.cu -- combine receive (weighted average accumulated on the
// receiving side), the grouped-GEMM stand-in, and the element-wise e4m3
// encoder, after "Enabling trillion-parameter models on AWS EFA", section
// "Dispatch and combine" (combine reads the receive buffer and accumulates
// each token's weighted average into the output).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "bf16.cuh"
#include "common.cuh"
#include "launch.h"

namespace moe {

// ------------------------------------------------------------ combine reduce
//
// One small block per token, or per part of a token's rows when the batch
// is too small to fill the GPU (grid-stride over blocks).  Threads 0..R-1
// resolve where each of the token's R rows sits (rank p = e/Er, row
// csend_off[p][s] + slot - send_off[s][p]) into shared memory; then every
// thread takes 16-byte chunks of the row, issues the R loads, and folds them
// into fp32 accumulators with one fused multiply-add per slot in slot order
// k = 0..R-1, rounding once to bf16 at the end.
constexpr int kReduceGroup = 8;  // row loads kept in flight per chunk
// Fewest blocks per token in the fused combine (small batches take more,
// see token_split): two, each a contiguous half of every row, when a half
// still gives every thread at least one 16-byte chunk per row (H >= 4096
// with 256 threads).  On the DSv3 EP16 combine two blocks per token
// measured 84.6 us against 86.7 us with whole tokens (finer work evens out
// the last wave of blocks); 4 or 8 were no better; on H = 2048 rows the
// split would leave half of every block idle.
static int combine_split(int H, int threads) { return (H >> 3) >= 2 * threads ? 2 : 1; }

// Threads per block of the fused combine: kGatherThreads, or half as many
// for rows of at most MOE_GATHER_NARROW_H elements, so that a short row
// (2048 elements: 256 16-byte chunks) is still split over two blocks, each
// thread one chunk of every row.  On the Qwen3-shaped EP16 combine
// (H = 2048) that measured 94.5 against 98.1 us and the layer graph 153.2
// against 156.5 us; on 7168-element rows 128 threads were slower (Kimi-K2
// EP32 layer 261 against 257 us).
#ifndef MOE_GATHER_NARROW_H
#define MOE_GATHER_NARROW_H 2048
#endif
constexpr int kGatherNarrow = kGatherThreads / 2;
static int gather_threads(int H) {
    return H <= MOE_GATHER_NARROW_H && kGatherNarrow >= 32 ? kGatherNarrow : kGatherThreads;
}

// kLL: the rows come from the low-latency layout, row ll_row[s][t][k] of
// `csend` (there y_ll), instead of the combine send buffers.
template <bool kLL>
__global__ void __launch_bounds__(kReduceThreads)
    k_combine_reduce(int N, int T, int E, int R, int H, int cap, int split, long long tok0,
                     long long tok1,
                     const uint16_t *__restrict__ csend, const int32_t *__restrict__ idx,
                     const float *__restrict__ w, const int32_t *__restrict__ slot_row,
                     const int32_t *__restrict__ send_off, const int32_t *__restrict__ csend_off,
                     const int32_t *__restrict__ ll_row, uint16_t *__restrict__ out) {
    __shared__ long long src[MOE_MAX_TOPK];  // element offset of row k in csend, -1: skip
    __shared__ float wk[MOE_MAX_TOPK];
    const int Er = E / N, cpr = H >> 3;
    // `split` blocks share a token, each a contiguous part of its rows
    const int per = (cpr + split - 1) / split;
    const long long nblk = (tok1 - tok0) * split;
    for (long long blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const long long tok = tok0 + blk / split;
        const int c0 = (int)(blk - (tok - tok0) * split) * per, c1 = min(cpr, c0 + per);
        const int s = (int)div_nonneg(tok, T);
        if (threadIdx.x < R) {
            const int k = threadIdx.x;
            long long o = -1;
            if constexpr (kLL) {
                const int row = __ldg(ll_row + tok * R + k);
                if (row >= 0) o = (long long)row * H;
            } else {
                const int e = __ldg(idx + tok * R + k);
                const int sl = __ldg(slot_row + tok * R + k);
                if ((unsigned)e < (unsigned)E && sl >= 0) {
                    const int p = e / Er;
                    const int c = __ldg(csend_off + (size_t)p * (N + 1) + s) +
                                  (sl - __ldg(send_off + (size_t)s * (N + 1) + p));
                    if (c >= 0 && c < cap) o = ((long long)p * cap + c) * H;
                }
            }
            src[k] = o;
            wk[k] = __ldg(w + tok * R + k);
        }
        __syncthreads();
        for (int part = c0 + threadIdx.x; part < c1; part += blockDim.x) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k0 = 0; k0 < R; k0 += kReduceGroup) {
                uint4 v[kReduceGroup];
#pragma unroll
                for (int u = 0; u < kReduceGroup; ++u) {
                    const int k = k0 + u;
                    if (k < R && src[k] >= 0)
                        v[u] = __ldcs(reinterpret_cast<const uint4 *>(csend + src[k]) + part);
                }
#pragma unroll
                for (int u = 0; u < kReduceGroup; ++u) {
                    const int k = k0 + u;
                    if (k < R && src[k] >= 0) fma8(acc, wk[k], v[u]);
                }
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            reinterpret_cast<uint4 *>(out + tok * H)[part] = o;
        }
        __syncthreads();
    }
}

// Blocks per token for the reduce: as many as a wave of resident blocks
// holds per token (rounded down, so a batch that fills the wave keeps one
// block per token), at most one 16-byte chunk per thread of every row.  On
// the DSv3 EP16 shape with 16 tokens the low-latency combine took 25.2 us
// with one block per token, its 64 threads walking 14 chunks of each row in
// turn.
template <bool kLL>
static cudaError_t reduce_grid(long long ntok, int H, int *split, int *grid) {
    static LaunchMemo memo;
    int occ = 1;
    const cudaError_t err = memo.get(0, &occ, [](int *v) {
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            v, k_combine_reduce<kLL>, kReduceThreads, 0);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    *split = token_split(ntok, H, kReduceThreads, occ, 1);
    const long long nblk = ntok * *split;
    *grid = (int)(nblk < (1LL << 30) ? nblk : (1LL << 30));
    return cudaSuccess;
}

cudaError_t launch_combine_reduce(const moe_shape &sh, int cap, const uint16_t *csend,
                                  const int32_t *idx, const float *w, const int32_t *slot_row,
                                  const int32_t *send_off, const int32_t *csend_off,
                                  uint16_t *out, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    if (ntok <= 0) return cudaSuccess;
    int split = 1, grid = 1;
    const cudaError_t err = reduce_grid<false>(ntok, sh.H, &split, &grid);
    if (err != cudaSuccess) return err;
    return launch_kernel(k_combine_reduce<false>, dim3((unsigned)grid), dim3(kReduceThreads), 0,
                         st, sh.N, sh.T, sh.E, sh.R, sh.H, cap, split, 0LL, ntok, csend, idx, w,
                         slot_row, send_off, csend_off, (const int32_t *)nullptr, out);
}

cudaError_t launch_combine_ll(const moe_shape &sh, const uint16_t *y_ll, const float *w,
                              const int32_t *ll_row, uint16_t *out, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    if (ntok <= 0) return cudaSuccess;
    int split = 1, grid = 1;
    const cudaError_t err = reduce_grid<true>(ntok, sh.H, &split, &grid);
    if (err != cudaSuccess) return err;
    return launch_kernel(k_combine_reduce<true>, dim3((unsigned)grid), dim3(kReduceThreads), 0,
                         st, sh.N, sh.T, sh.E, sh.R, sh.H, 0, split, 0LL, ntok, y_ll,
                         (const int32_t *)nullptr, w, (const int32_t *)nullptr,
                         (const int32_t *)nullptr, (const int32_t *)nullptr, ll_row, out);
}

// ------------------------------------------------------------ fused combine
//
// combine_send and combine_recv in one pass.  For token t of rank s and slot
// k (expert e on rank p), the expert output sits at grouped row
// g = seg_off[p][j][s] + (slot - expert_send_off[s][e]) of y and belongs at
// combine row c = csend_off[p][s] + (slot - send_off[s][p]).  The block
// reads each of the token's R rows once from y, writes it to its csend row
// (so the combine send buffer is produced exactly as by moe_combine_send) and
// folds the same values into the fp32 accumulator in slot order, as
// moe_combine_recv would after reading them back.  A row whose grouped
// position was dropped is written as zeros and contributes w * 0.
// KR: 0, slots read from shared memory; else R <= KR slots held in registers.
// kThreads: the block size it is launched with.
template <int KR, int kThreads>
__global__ void __launch_bounds__(kThreads)
    k_combine_fused(int N, int T, int E, int R, int H, int cap, int split,
                    const uint16_t *__restrict__ y,
                    const int32_t *__restrict__ idx, const float *__restrict__ w,
                    const int32_t *__restrict__ slot_row, const int32_t *__restrict__ eso,
                    const int32_t *__restrict__ seg_off, const int32_t *__restrict__ send_off,
                    const int32_t *__restrict__ csend_off, uint16_t *__restrict__ csend,
                    uint16_t *__restrict__ out) {
    __shared__ long long ysrc[MOE_MAX_TOPK];  // element offset of the row in y, -1: zeros
    __shared__ long long cdst[MOE_MAX_TOPK];  // element offset in csend, -1: not sent
    __shared__ float wk[MOE_MAX_TOPK];
    const int Er = E / N, cpr = H >> 3;
    const long long ntok = (long long)N * T;
    // `split` blocks share a token, each a contiguous part of its rows
    const int per = (cpr + split - 1) / split;
    for (long long blk = blockIdx.x; blk < ntok * split; blk += gridDim.x) {
        const long long tok = blk / split;
        const int c0 = (int)(blk - tok * split) * per, c1 = min(cpr, c0 + per);
        const int s = (int)div_nonneg(tok, T);
        if (threadIdx.x < R) {
            const int k = threadIdx.x;
            const int e = __ldg(idx + tok * R + k);
            const int sl = __ldg(slot_row + tok * R + k);
            long long yo = -1, co = -1;
            if ((unsigned)e < (unsigned)E && sl >= 0) {
                const int p = e / Er, j = e - p * Er;
                const int c = __ldg(csend_off + (size_t)p * (N + 1) + s) +
                              (sl - __ldg(send_off + (size_t)s * (N + 1) + p));
                if (c >= 0 && c < cap) {
                    co = ((long long)p * cap + c) * H;
                    const int g = __ldg(seg_off + ((size_t)p * Er + j) * N + s) +
                                  (sl - __ldg(eso + (size_t)s * (E + 1) + e));
                    if (g >= 0 && g < cap) yo = ((long long)p * cap + g) * H;
                }
            }
            ysrc[k] = yo;
            cdst[k] = co;
            wk[k] = __ldg(w + tok * R + k);
        }
        __syncthreads();
        if constexpr (KR > 0) {
            const uint4 *ys[KR];
            uint4 *cs[KR];
            float wr[KR];
#pragma unroll
            for (int u = 0; u < KR; ++u) {
                const bool on = u < R;
                ys[u] = on && ysrc[u] >= 0 ? reinterpret_cast<const uint4 *>(y + ysrc[u]) : nullptr;
                cs[u] = on && cdst[u] >= 0 ? reinterpret_cast<uint4 *>(csend + cdst[u]) : nullptr;
                wr[u] = on ? wk[u] : 0.0f;
            }
            for (int part = c0 + threadIdx.x; part < c1; part += blockDim.x) {
                uint4 v[KR];
#pragma unroll
                for (int u = 0; u < KR; ++u)
                    v[u] = ys[u] ? __ldcs(ys[u] + part) : make_uint4(0, 0, 0, 0);
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u = 0; u < KR; ++u) {
                    if (cs[u]) {
                        cs[u][part] = v[u];
                        fma8(acc, wr[u], v[u]);
                    }
                }
                uint4 o;
                o.x = pack_bf16x2(acc[0], acc[1]);
                o.y = pack_bf16x2(acc[2], acc[3]);
                o.z = pack_bf16x2(acc[4], acc[5]);
                o.w = pack_bf16x2(acc[6], acc[7]);
                reinterpret_cast<uint4 *>(out + tok * H)[part] = o;
            }
        } else {
            for (int part = c0 + threadIdx.x; part < c1; part += blockDim.x) {
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int k0 = 0; k0 < R; k0 += kReduceGroup) {
                    uint4 v[kReduceGroup];
#pragma unroll
                    for (int u = 0; u < kReduceGroup; ++u) {
                        const int k = k0 + u;
                        v[u] = make_uint4(0, 0, 0, 0);
                        if (k < R && ysrc[k] >= 0)
                            v[u] = __ldcs(reinterpret_cast<const uint4 *>(y + ysrc[k]) + part);
                    }
#pragma unroll
                    for (int u = 0; u < kReduceGroup; ++u) {
                        const int k = k0 + u;
                        if (k < R && cdst[k] >= 0) {
                            reinterpret_cast<uint4 *>(csend + cdst[k])[part] = v[u];
                            fma8(acc, wk[k], v[u]);
                        }
                    }
                }
                uint4 o;
                o.x = pack_bf16x2(acc[0], acc[1]);
                o.y = pack_bf16x2(acc[2], acc[3]);
                o.z = pack_bf16x2(acc[4], acc[5]);
                o.w = pack_bf16x2(acc[6], acc[7]);
                reinterpret_cast<uint4 *>(out + tok * H)[part] = o;
            }
        }
        __syncthreads();
    }
}

cudaError_t launch_combine_fused(const moe_shape &sh, int cap, const uint16_t *y,
                                 const int32_t *idx, const float *w, const int32_t *slot_row,
                                 const int32_t *eso, const int32_t *seg_off,
                                 const int32_t *send_off, const int32_t *csend_off,
                                 uint16_t *csend, uint16_t *out, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    if (ntok <= 0) return cudaSuccess;
    const int kr = sh.R <= 8 ? 8 : 0;
    const int threads = gather_threads(sh.H);
    const bool narrow = threads != kGatherThreads;
    auto kern = kr ? (narrow ? k_combine_fused<8, kGatherNarrow> : k_combine_fused<8, kGatherThreads>)
                   : (narrow ? k_combine_fused<0, kGatherNarrow> : k_combine_fused<0, kGatherThreads>);
    static LaunchMemo memo;
    int occ = 1;
    const cudaError_t err = memo.get(kr * 2 + (narrow ? 1 : 0), &occ, [&](int *v) {
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, 0);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    // small batches: more blocks per token, as for the reduce
    const int split = token_split(ntok, sh.H, threads, occ, combine_split(sh.H, threads));
    const long long nblk = ntok * split;
    const int grid = (int)(nblk < (1LL << 30) ? nblk : (1LL << 30));
    return launch_kernel(kern, dim3((unsigned)grid), dim3(threads), 0, st, sh.N, sh.T, sh.E,
                         sh.R, sh.H, cap, split, y, idx, w, slot_row, eso, seg_off, send_off,
                         csend_off, csend, out);
}

// ------------------------------------------------------------ expert stand-in
//
// Not part of the timed path.  One warp per grouped row (grid-stride over
// N*cap rows, rows past the received count skipped); y = bf16_rn((dq * scale)
// * s_e) with fp32 multiplies.
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(h));
}

__global__ void __launch_bounds__(256)
    k_expert_standin(int N, int E, int H, int cap, int mode, const uint8_t *__restrict__ grp_q,
                     const float *__restrict__ grp_s, const int32_t *__restrict__ grp_off,
                     uint16_t *__restrict__ y) {
    const int lane = threadIdx.x & 31, Er = E / N, Sb = H >> 7;
    const long long nrows = (long long)N * cap;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         row < nrows; row += nwarps) {
        const int r = (int)(row / cap), g = (int)(row - (long long)r * cap);
        const int32_t *go = grp_off + (size_t)r * (Er + 1);
        if (g >= __ldg(go + Er)) continue;
        const int e = r * Er + find_run(go, Er, g);
        const float se = mode == 0 ? 1.0f : (e % 3 == 0 ? 0.5f : (e % 3 == 1 ? 1.0f : 2.0f));
        const uint8_t *q = grp_q + row * H;
        for (int c = lane; c < (H >> 4); c += 32) {
            const uint4 qv = *reinterpret_cast<const uint4 *>(q + c * 16);
            const float sc = __ldg(grp_s + row * Sb + (c >> 3));
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t o[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t word = qw[u >> 1] >> ((u & 1) * 16);
                const float a = __fmul_rn(__fmul_rn(e4m3_to_float((uint8_t)(word & 0xff)), sc), se);
                const float b =
                    __fmul_rn(__fmul_rn(e4m3_to_float((uint8_t)((word >> 8) & 0xff)), sc), se);
                o[u] = pack_bf16x2(a, b);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(y + row * H + c * 16);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
}

cudaError_t launch_expert_standin(const moe_shape &sh, int cap, int mode, const uint8_t *grp_q,
                                  const float *grp_s, const int32_t *grp_off, uint16_t *y,
                                  cudaStream_t st) {
    const long long nrows = (long long)sh.N * cap;
    if (nrows == 0) return cudaSuccess;
    const long long need = (nrows + 7) / 8;
    const long long cap_blocks = (long long)sm_count() * 8;
    const int grid = (int)(need < cap_blocks ? need : cap_blocks);
    k_expert_standin<<<grid, 256, 0, st>>>(sh.N, sh.E, sh.H, cap, mode, grp_q, grp_s, grp_off, y);
    return cudaGetLastError();
}

// Stand-in over the low-latency layout: row `row` is in region
// reg = row / T = e*N + s (expert e); it holds data when row % T <
// min(count[reg], T).
__global__ void __launch_bounds__(256)
    k_expert_standin_ll(int N, int T, int E, int H, int mode, const uint8_t *__restrict__ ll_q,
                        const float *__restrict__ ll_s, const int32_t *__restrict__ ll_count,
                        uint16_t *__restrict__ y) {
    const int lane = threadIdx.x & 31, Sb = H >> 7;
    const long long nrows = (long long)N * E * T;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         row < nrows; row += nwarps) {
        const long long reg = row / T;
        const int u = (int)(row - reg * T);
        if (u >= __ldg(ll_count + reg)) continue;
        const int e = (int)(reg / N);
        const float se = mode == 0 ? 1.0f : (e % 3 == 0 ? 0.5f : (e % 3 == 1 ? 1.0f : 2.0f));
        const uint8_t *q = ll_q + row * H;
        for (int c = lane; c < (H >> 4); c += 32) {
            const uint4 qv = *reinterpret_cast<const uint4 *>(q + c * 16);
            const float sc = __ldg(ll_s + row * Sb + (c >> 3));
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t o[8];
#pragma unroll
            for (int u2 = 0; u2 < 8; ++u2) {
                const uint32_t word = qw[u2 >> 1] >> ((u2 & 1) * 16);
                const float a = __fmul_rn(__fmul_rn(e4m3_to_float((uint8_t)(word & 0xff)), sc), se);
                const float b =
                    __fmul_rn(__fmul_rn(e4m3_to_float((uint8_t)((word >> 8) & 0xff)), sc), se);
                o[u2] = pack_bf16x2(a, b);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(y + row * H + c * 16);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
}

cudaError_t launch_expert_standin_ll(const moe_shape &sh, int mode, const uint8_t *ll_q,
                                     const float *ll_s, const int32_t *ll_count, uint16_t *y_ll,
                                     cudaStream_t st) {
    const long long nrows = (long long)sh.N * sh.E * sh.T;
    if (nrows == 0) return cudaSuccess;
    const long long need = (nrows + 7) / 8;
    const long long cap_blocks = (long long)sm_count() * 8;
    const int grid = (int)(need < cap_blocks ? need : cap_blocks);
    k_expert_standin_ll<<<grid, 256, 0, st>>>(sh.N, sh.T, sh.E, sh.H, mode, ll_q, ll_s, ll_count,
                                              y_ll);
    return cudaGetLastError();
}

// ------------------------------------------------------------ e4m3 encoder
//
// The same conversion as the quantiser (pairs through
// __nv_cvt_float2_to_fp8x2, saturating, round to nearest even).
__global__ void k_e4m3_encode(const float *__restrict__ v, uint8_t *__restrict__ out,
                              long long n) {
    const long long npairs = (n + 1) / 2;
    for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < npairs;
         p += (long long)gridDim.x * blockDim.x) {
        const long long i = 2 * p;
        const float a = v[i];
        const float b = i + 1 < n ? v[i + 1] : 0.0f;
        const uint32_t c =
            (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        out[i] = (uint8_t)(c & 0xff);
        if (i + 1 < n) out[i + 1] = (uint8_t)(c >> 8);
    }
}

cudaError_t launch_e4m3_encode(const float *v, uint8_t *out, int64_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const long long need = ((n + 1) / 2 + 255) / 256;
    const long long cap_blocks = (long long)sm_count() * 8;
    const int grid = (int)(need < cap_blocks ? need : cap_blocks);
    k_e4m3_encode<<<grid, 256, 0, st>>>(v, out, n);
    return cudaGetLastError();
}

}  // namespace moe
