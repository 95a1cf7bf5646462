// partial.cu -- the combine with send-side reduction: the alternative that
// "Enabling trillion-parameter models on AWS EFA" ("Evaluation:
// dispatch/combine latency", prefill) contrasts with its receive-side-only
// accumulation -- summing on the sending side cuts the bytes sent, at some
// cost in accuracy.
//
// Expert rank r sums, for each token (s, t) with experts on r, the weighted
// outputs of those experts (fp32 fused multiply-adds in slot order) and
// rounds the partial once to bf16: one row part[r][s][t] instead of one row
// per assignment.  The receiver adds its token's partials in ascending rank
// order in fp32 and rounds once more.
//
// One small block per token, or per part of a token's rows when the batch
// is too small to fill the GPU (grid-stride over blocks).  Warp 0 sorts the
// token's valid slots by (rank, slot) with one lane per slot, so each rank's
// slots are consecutive and its last slot closes the partial; then every
// thread takes 16-byte chunks of the row.
#include "bf16.cuh"
#include "common.cuh"
#include "launch.h"

namespace moe {

static_assert(kReduceThreads >= 32 && kGatherThreads >= 32, "warp 0 sorts the slots");

// The sending side and the one-pass form take the fused combine's block
// shape: half of kGatherThreads for rows of at most MOE_GATHER_NARROW_H
// elements, and two blocks per token when half of every row still gives
// each thread a 16-byte chunk.  Against 256 threads and one block per
// token: the Qwen3-shaped EP16 one-pass form 93.4 against 95.8 us (layer
// graph 151.1 against 153.1), DSv3 EP16 79.4 against 81.5 (layer 130.8
// against 132.7), Kimi-K2 unchanged.
#ifndef MOE_GATHER_NARROW_H
#define MOE_GATHER_NARROW_H 2048
#endif
static_assert(kGatherThreads / 2 >= 32, "the narrow block still holds warp 0's sort");

enum class PartialMode { kSend, kRecv, kFused };

template <PartialMode kMode, int KR>  // KR > 0: R <= KR rows in registers; 0: any R
__global__ void __launch_bounds__(kGatherThreads > kReduceThreads ? kGatherThreads
                                                                   : kReduceThreads)
    k_combine_partial(int N, int T, int E, int R, int H, int cap, int split,
                      const uint16_t *__restrict__ y,
                      const int32_t *__restrict__ idx, const float *__restrict__ w,
                      const int32_t *__restrict__ slot_row, const int32_t *__restrict__ eso,
                      const int32_t *__restrict__ seg_off, uint16_t *__restrict__ pbuf,
                      uint16_t *__restrict__ out) {
    constexpr bool kReadY = kMode != PartialMode::kRecv;
    constexpr bool kWriteOut = kMode != PartialMode::kSend;
    // the token's valid slots in (rank, slot) order: y row (element offset,
    // -1: dropped, reads as zeros), weight, partial row (element offset),
    // and whether the slot is its rank's last
    __shared__ long long oy[MOE_MAX_TOPK], op[MOE_MAX_TOPK];
    __shared__ float ow[MOE_MAX_TOPK];
    __shared__ int oend[MOE_MAX_TOPK];
    __shared__ int nval;
    const int Er = E / N, cpr = H >> 3;
    const long long ntok = (long long)N * T;
    // `split` blocks share a token, each a contiguous part of its rows
    const int per = (cpr + split - 1) / split;
    for (long long blk = blockIdx.x; blk < ntok * split; blk += gridDim.x) {
        const long long tok = blk / split;
        const int c0 = (int)(blk - tok * split) * per, c1 = min(cpr, c0 + per);
        const int s = (int)div_nonneg(tok, T);
        const int t = (int)(tok - (long long)s * T);
        if (threadIdx.x < 32) {
            const int k = threadIdx.x;
            int p = -1;
            long long yo = -1;
            float wk = 0.0f;
            if (k < R) {
                const int e = __ldg(idx + tok * R + k);
                const int sl = __ldg(slot_row + tok * R + k);
                if ((unsigned)e < (unsigned)E && sl >= 0) {
                    p = e / Er;
                    if (kReadY) {
                        const int j = e - p * Er;
                        const int g = __ldg(seg_off + ((size_t)p * Er + j) * N + s) +
                                      (sl - __ldg(eso + (size_t)s * (E + 1) + e));
                        if (g >= 0 && g < cap) yo = ((long long)p * cap + g) * H;
                        wk = __ldg(w + tok * R + k);
                    }
                }
            }
            int pos = 0;
            bool last = true;
            for (int q = 0; q < R; ++q) {
                const int pq = __shfl_sync(kFull, p, q);
                if (p >= 0 && pq >= 0 && (pq < p || (pq == p && q < k))) ++pos;
                if (p >= 0 && pq == p && q > k) last = false;
            }
            const int nv = __popc(__ballot_sync(kFull, p >= 0));
            if (p >= 0) {
                oy[pos] = yo;
                ow[pos] = wk;
                op[pos] = (((long long)p * N + s) * T + t) * H;
                oend[pos] = last;
            }
            if (k == 0) nval = nv;
        }
        __syncthreads();
        const int nv = nval;
        uint4 *orow = reinterpret_cast<uint4 *>(out + tok * H);
        if constexpr (KR > 0) {
            const uint4 *ys[KR];
            uint4 *ps[KR];
            float wr[KR];
#pragma unroll
            for (int u = 0; u < KR; ++u) {
                const bool on = u < nv;
                ys[u] = kReadY && on && oy[u] >= 0 ? reinterpret_cast<const uint4 *>(y + oy[u])
                                                    : nullptr;
                ps[u] = on && oend[u] ? reinterpret_cast<uint4 *>(pbuf + op[u]) : nullptr;
                wr[u] = on ? ow[u] : 0.0f;
            }
            for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
                float acc_o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if constexpr (kReadY) {
                    uint4 v[KR];
#pragma unroll
                    for (int u = 0; u < KR; ++u)
                        v[u] = ys[u] ? __ldcs(ys[u] + c) : make_uint4(0, 0, 0, 0);
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int u = 0; u < KR; ++u) {
                        if (u < nv) {
                            fma8(acc, wr[u], v[u]);
                            if (ps[u]) {
                                const uint4 pk = pack_bf16x8(acc);
                                ps[u][c] = pk;
                                if (kWriteOut) add8(acc_o, pk);
#pragma unroll
                                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                            }
                        }
                    }
                } else {
                    uint4 v[KR];
#pragma unroll
                    for (int u = 0; u < KR; ++u)
                        v[u] = ps[u] ? __ldcs(ps[u] + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int u = 0; u < KR; ++u)
                        if (ps[u]) add8(acc_o, v[u]);
                }
                if (kWriteOut) orow[c] = pack_bf16x8(acc_o);
            }
        } else {
            for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
                float acc_o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int u = 0; u < nv; ++u) {
                    uint4 *prow = reinterpret_cast<uint4 *>(pbuf + op[u]);
                    if constexpr (kReadY) {
                        const uint4 v = oy[u] >= 0
                                            ? __ldcs(reinterpret_cast<const uint4 *>(y + oy[u]) + c)
                                            : make_uint4(0, 0, 0, 0);
                        fma8(acc, ow[u], v);
                        if (oend[u]) {
                            const uint4 pk = pack_bf16x8(acc);
                            prow[c] = pk;
                            if (kWriteOut) add8(acc_o, pk);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                        }
                    } else if (oend[u]) {
                        add8(acc_o, __ldcs(prow + c));
                    }
                }
                if (kWriteOut) orow[c] = pack_bf16x8(acc_o);
            }
        }
        __syncthreads();
    }
}

template <PartialMode kMode>
static cudaError_t launch_partial(const moe_shape &sh, int cap, const uint16_t *y,
                                  const int32_t *idx, const float *w, const int32_t *slot_row,
                                  const int32_t *eso, const int32_t *seg_off, uint16_t *pbuf,
                                  uint16_t *out, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    if (ntok <= 0) return cudaSuccess;
    const int kr = sh.R <= 8 ? 8 : 0;
    auto kern = kr ? k_combine_partial<kMode, 8> : k_combine_partial<kMode, 0>;
    // the receiving side only reads rows: the smaller block (see bf16.cuh)
    int threads = kReduceThreads, least = 1;
    if (kMode != PartialMode::kRecv) {
        threads = sh.H <= MOE_GATHER_NARROW_H ? kGatherThreads / 2 : kGatherThreads;
        least = (sh.H >> 3) >= 2 * threads ? 2 : 1;
    }
    static LaunchMemo memo;
    int occ = 1;
    const cudaError_t err = memo.get(kr * 1024 + threads, &occ, [&](int *v) {
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, 0);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    const int split = token_split(ntok, sh.H, threads, occ, least);
    const long long nblk = ntok * split;
    const int grid = (int)(nblk < (1LL << 30) ? nblk : (1LL << 30));
    return launch_kernel(kern, dim3((unsigned)grid), dim3(threads), 0, st, sh.N, sh.T,
                         sh.E, sh.R, sh.H, cap, split, y, idx, w, slot_row, eso, seg_off, pbuf,
                         out);
}

cudaError_t launch_combine_partial_send(const moe_shape &sh, int cap, const uint16_t *y,
                                        const int32_t *idx, const float *w,
                                        const int32_t *slot_row, const int32_t *eso,
                                        const int32_t *seg_off, uint16_t *pbuf, cudaStream_t st) {
    return launch_partial<PartialMode::kSend>(sh, cap, y, idx, w, slot_row, eso, seg_off, pbuf,
                                              nullptr, st);
}

cudaError_t launch_combine_partial_recv(const moe_shape &sh, const uint16_t *pbuf,
                                        const int32_t *idx, const int32_t *slot_row,
                                        uint16_t *out, cudaStream_t st) {
    return launch_partial<PartialMode::kRecv>(sh, 0, nullptr, idx, nullptr, slot_row, nullptr,
                                              nullptr, const_cast<uint16_t *>(pbuf), out, st);
}

cudaError_t launch_combine_partial(const moe_shape &sh, int cap, const uint16_t *y,
                                   const int32_t *idx, const float *w, const int32_t *slot_row,
                                   const int32_t *eso, const int32_t *seg_off, uint16_t *pbuf,
                                   uint16_t *out, cudaStream_t st) {
    return launch_partial<PartialMode::kFused>(sh, cap, y, idx, w, slot_row, eso, seg_off, pbuf,
                                               out, st);
}

}  // namespace moe
