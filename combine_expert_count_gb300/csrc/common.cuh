// common.cuh -- device helpers shared by the libmoeroute kernels (sm_103a).
//
// Warp / block scans, the status word, and thin inline-PTX wrappers for the
// mbarrier and bulk-async-copy (TMA, non-tensor) loads the quantiser uses and
// the acquire / release flag accesses of the signalled dispatch.  Every wait
// on an mbarrier is bounded by a cycle budget and reports MOE_ST_TIMEOUT
// instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moeroute.h"

namespace moe {

constexpr unsigned kFull = 0xffffffffu;

// ~1 s at GB300 clocks: far beyond any legitimate copy latency.
constexpr long long kWaitCycles = 2000000000LL;

__device__ __forceinline__ void flag(int32_t *status, int bits) { atomicOr(status, bits); }

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// Inclusive scan over the block (blockDim.x a multiple of 32, <= 1024).
// `wsum` is __shared__ int[32]; `*total` (shared) receives the block total.
// Contains __syncthreads(); every thread of the block must call it.
__device__ __forceinline__ int block_inclusive_scan(int v, int *wsum, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = warp_inclusive_scan(v);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? wsum[lane] : 0;
        int wi = warp_inclusive_scan(w);
        if (lane < nw) wsum[lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return incl + wsum[warp];
}

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (clock64() - t0 < kWaitCycles)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both 16-B aligned);
// completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// GPU-scope acquire load / release store of a 32-bit flag.
__device__ __forceinline__ int ld_acquire(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int32_t *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Address of `p` (this block's shared memory) in the shared memory of
// cluster block `rank`, and a 32-bit load from such an address.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ int ld_dsmem(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------------ misc

// Round a shared-memory pointer up to a 128-byte boundary.
template <class T>
__device__ __forceinline__ T *align128(T *p) {
    return reinterpret_cast<T *>((reinterpret_cast<uintptr_t>(p) + 127) &
                                 ~static_cast<uintptr_t>(127));
}

// a / b for non-negative a, b > 0: a 32-bit division when both fit (a 64-bit
// division costs dozens of instructions).
__device__ __forceinline__ long long div_nonneg(long long a, long long b) {
    if (a <= 0xffffffffLL && b <= 0xffffffffLL)
        return (long long)((unsigned)a / (unsigned)b);
    return a / b;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Largest e in [0, E) with off[e] <= i, given off[0] <= i < off[E] and off
// non-decreasing (an exclusive scan of counts).
__device__ __forceinline__ int find_run(const int32_t *__restrict__ off, int E, int i) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(off + mid) <= i)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Launch `kern` on `st` with the given geometry.
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same as a cooperative launch: every CTA of the grid is resident at
// once (the launch fails instead if they cannot be), so CTAs may wait on
// flags that other CTAs of the grid set.
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel_coresident(void (*kern)(KArgs...), dim3 grid, dim3 block,
                                            size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace moe
