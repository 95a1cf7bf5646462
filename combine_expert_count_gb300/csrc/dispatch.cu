// dispatch.cu -- dispatch send: block-scaled fp8 quantisation fused with the
// pack into contiguous per-peer send buffers, after "Enabling
// trillion-parameter models on AWS EFA", sections "Dispatch and combine"
// (pack once the offsets are known) and "Evaluation: dispatch/combine
// latency" (block-scaled fp8 dispatch).
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

// ------------------------------------------------------------ quant + pack
//
// One thread per 16 consecutive elements of a token row: two 16-byte loads
// of x, 8 lanes per 128-element block (amax by xor-shuffles within the
// group), scale = amax/448 and q = e4m3_satfinite_rn(x/scale) with IEEE fp32
// divisions, then one 16-byte store into each of the token's R send rows.
// A warp covers 512 contiguous bytes of a row, so every store is a full
// coalesced line.
constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t cvt_pair(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__global__ void __launch_bounds__(kQuantThreads)
    k_quant_pack(int T, int R, int H, long long nchunks, const uint16_t *__restrict__ x,
                 const int32_t *__restrict__ slot_row, uint8_t *__restrict__ send_q,
                 float *__restrict__ send_s, int32_t *__restrict__ send_tok) {
    const int lane = threadIdx.x & 31;
    const int cpr = H >> 4;  // 16-element chunks per row
    const int Sb = H >> 7;
    const long long TR = (long long)T * R;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c0 = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); c0 < nchunks;
         c0 += stride) {
        const long long c = c0 + lane;
        const bool in = c < nchunks;
        const long long tok = in ? c / cpr : 0;
        const int part = in ? (int)(c - tok * cpr) : 0;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (in) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + tok * H + (long long)part * 16);
            a = __ldcs(src);
            b = __ldcs(src + 1);
        }
        float f[16];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            f[2 * u] = bf16_lo(w[u]);
            f[2 * u + 1] = bf16_hi(w[u]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int u = 0; u < 16; ++u) amax = fmaxf(amax, fabsf(f[u]));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
        const float scale = __fdiv_rn(amax, 448.0f);
        uint4 q = make_uint4(0, 0, 0, 0);
        if (amax > 0.0f) {
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t lo = cvt_pair(__fdiv_rn(f[4 * u], scale), __fdiv_rn(f[4 * u + 1], scale));
                const uint32_t hi =
                    cvt_pair(__fdiv_rn(f[4 * u + 2], scale), __fdiv_rn(f[4 * u + 3], scale));
                o[u] = lo | (hi << 16);
            }
            q = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (in) {
            const long long s = tok / T;
            const int t = (int)(tok - s * T);
            const int32_t *sl = slot_row + tok * R;
            for (int k = 0; k < R; ++k) {
                const int sr = __ldg(sl + k);
                if (sr < 0 || sr >= TR) continue;  // skipped assignment
                const long long row = s * TR + sr;
                *reinterpret_cast<uint4 *>(send_q + row * H + (long long)part * 16) = q;
                if ((part & 7) == 0) send_s[row * Sb + (part >> 3)] = scale;
                if (part == 0) send_tok[row] = t;
            }
        }
    }
}

cudaError_t launch_quant_pack(const moe_shape &sh, const uint16_t *x, const int32_t *slot_row,
                              uint8_t *send_q, float *send_s, int32_t *send_tok, cudaStream_t st) {
    const long long nchunks = (long long)sh.N * sh.T * (sh.H / 16);
    if (nchunks == 0) return cudaSuccess;
    const long long need = (nchunks + kQuantThreads - 1) / kQuantThreads;
    const long long cap_blocks = (long long)sm_count() * (2048 / kQuantThreads);
    const int grid = (int)(need < cap_blocks ? need : cap_blocks);
    k_quant_pack<<<grid, kQuantThreads, 0, st>>>(sh.T, sh.R, sh.H, nchunks, x, slot_row, send_q,
                                                 send_s, send_tok);
    return cudaGetLastError();
}

}  // namespace moe
