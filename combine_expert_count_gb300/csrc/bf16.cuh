// bf16.cuh -- bf16 <-> fp32 helpers of the combine kernels: round-to-nearest-
// even packing of two fp32 values, and eight fused multiply-adds of a weight
// into fp32 accumulators from a 16-byte vector of bf16.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

#ifndef MOE_REDUCE_THREADS
#define MOE_REDUCE_THREADS 64
#endif
#ifndef MOE_GATHER_THREADS
#define MOE_GATHER_THREADS 256
#endif

namespace moe {

// Threads per token block.  Kernels that only read a token's rows and write
// its output (moe_combine_recv, moe_combine_ll, the receiving side of the
// send-side reduction) use 64: a 2048-token batch is one wave of resident
// blocks.  Kernels that also write every row they read (moe_combine, the
// sending side of the send-side reduction) use 256, each step covering a
// 4 KB stretch of every row: on the DSv3 EP16 combine that measured 86.7 us
// against 90.8 us with 64 threads (192, 384 and 512 were no better; with
// two blocks per token, 160, 224 and 448 measured 86.7, 84.6 and 94.9 us
// against 84.6, and 224 made the sending side of the send-side reduction
// 2 us slower), while the read-only reduce measured 39.4 us with 64 threads
// and 44.9 us with 256.
constexpr int kReduceThreads = MOE_REDUCE_THREADS;
constexpr int kGatherThreads = MOE_GATHER_THREADS;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&a)[8]) {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                      pack_bf16x2(a[6], a[7]));
}

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4 &v) {
    acc[0] = __fmaf_rn(w, bf16_lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(w, bf16_hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(w, bf16_lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(w, bf16_hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(w, bf16_lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(w, bf16_hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(w, bf16_lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(w, bf16_hi(v.w), acc[7]);
}

// acc += the eight bf16 values of v (fp32 additions, round to nearest).
__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v) {
    acc[0] = __fadd_rn(acc[0], bf16_lo(v.x));
    acc[1] = __fadd_rn(acc[1], bf16_hi(v.x));
    acc[2] = __fadd_rn(acc[2], bf16_lo(v.y));
    acc[3] = __fadd_rn(acc[3], bf16_hi(v.y));
    acc[4] = __fadd_rn(acc[4], bf16_lo(v.z));
    acc[5] = __fadd_rn(acc[5], bf16_hi(v.z));
    acc[6] = __fadd_rn(acc[6], bf16_lo(v.w));
    acc[7] = __fadd_rn(acc[7], bf16_hi(v.w));
}

}  // namespace moe
