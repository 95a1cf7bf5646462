// route.cu -- per-expert counting, exclusive scans and the routing-info
// exchange ("Enabling trillion-parameter models on AWS EFA", sections "Send
// and receive buffers" and "Dispatch and combine").
//
// k_route_count: one 1024-thread block per rank, as the page describes
//   (counts accumulated in shared memory inside a single block, then a
//   cumulative sum), and the stable slot of every (t, k) (see route_sender).
//   Each warp counts into a shared-memory table row of its own, so the counts
//   need no atomics, and the slots follow from the same tables.
//
// k_exchange: one block per receiver; a block scan over the Er*N counts in
//   (local expert, sender) order gives seg_off / grp_off / m_sizes, and a
//   second scan over senders gives csend_off.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "rank.cuh"

// Both routing kernels run 1024-thread blocks and the host refuses E above
// MOE_MAX_EXPERTS (1024), so every expert owns one thread of the block and the
// expert scan of sender_count is a single block scan (its kOneChunk form).
#ifndef MOE_ROUTE_REG_RANKS
#define MOE_ROUTE_REG_RANKS 1
#endif

namespace moe {

constexpr int kRouteThreads = 1024;

// Shared memory of the sender role: base ([E+1] ints: the exclusive scan of
// the counts, then the total) and the per-warp count table ([32 warps][E]).
static size_t route_smem(int E) { return ((size_t)E * 33 + 1) * sizeof(int); }

// Sender role, part 2: expert_count, expert_send_off and send_off from
// shared memory (`counts`), and the stable slots (`slots`).
__device__ __forceinline__ void sender_write(int N, int T, int E, int R,
                                             const int32_t *__restrict__ idx,
                                             int32_t *__restrict__ cnt_out,
                                             int32_t *__restrict__ send_off,
                                             int32_t *__restrict__ eso_out,
                                             int32_t *__restrict__ slot_row, const int *smem,
                                             const int (&rk)[kAhead], const SenderShare &sh,
                                             bool counts, bool slots) {
    const int *base = smem;
    const int s = blockIdx.x, tid = threadIdx.x;
    const int TR = T * R, Er = E / N;
    if (counts) {
        for (int e = tid; e <= E; e += blockDim.x) {
            if (e < E) cnt_out[(size_t)s * E + e] = base[e + 1] - base[e];
            eso_out[(size_t)s * (E + 1) + e] = base[e];
        }
        for (int p = tid; p <= N; p += blockDim.x)
            send_off[(size_t)s * (N + 1) + p] = base[p < N ? p * Er : E];
    }
    if (!slots) return;
    // 3. slots: expert offset + earlier ids of the rank with the same expert
    int32_t *srow = slot_row + (size_t)s * TR;
    sender_ranks(T, E, R, s, idx, slot_row, smem, rk, sh,
                 [&](int i, int e, int u) { srow[i] = e >= 0 ? base[e] + u : -1; });
}

// Both parts of the sender role (the separate-call form).
__device__ __forceinline__ bool route_sender(int N, int T, int E, int R,
                                             const int32_t *__restrict__ idx,
                                             int32_t *__restrict__ cnt_out,
                                             int32_t *__restrict__ send_off,
                                             int32_t *__restrict__ eso_out,
                                             int32_t *__restrict__ slot_row, int *smem) {
    int rk[kAhead];
    SenderShare sh;
    const bool bad = sender_count<true, MOE_ROUTE_REG_RANKS>(N, T, E, R, blockIdx.x, idx, slot_row, smem, rk, sh);
    sender_write(N, T, E, R, idx, cnt_out, send_off, eso_out, slot_row, smem, rk, sh, true, true);
    return bad;
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route_count(int N, int T, int E, int R, const int32_t *__restrict__ idx,
                  int32_t *__restrict__ cnt_out, int32_t *__restrict__ send_off,
                  int32_t *__restrict__ eso_out, int32_t *__restrict__ slot_row,
                  int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    if (route_sender(N, T, E, R, idx, cnt_out, send_off, eso_out, slot_row, smem) &&
        threadIdx.x == 0)
        flag(status, MOE_ST_BAD_EXPERT);
}

// Receiver role of rank r = blockIdx.x given v = the count of run f = j*N + s
// (local expert j, sender s) for tid < F = Er*N, and w = the rows sender
// tid sends to r for tid < N.
__device__ __forceinline__ void route_receiver(int N, int E, int cap, int v, int w,
                                               int32_t *__restrict__ grp_off,
                                               int32_t *__restrict__ seg_off,
                                               int32_t *__restrict__ csend_off,
                                               int32_t *__restrict__ m_sizes,
                                               int32_t *__restrict__ status) {
    __shared__ int wsum[32];
    __shared__ int total;
    __shared__ int excl[MOE_MAX_EXPERTS + 1];
    const int r = blockIdx.x, tid = threadIdx.x, Er = E / N, F = Er * N;
    const int incl = block_inclusive_scan(v, wsum, &total);
    if (tid < F) {
        excl[tid] = incl - v;
        seg_off[(size_t)r * F + tid] = incl - v;  // [r][j][s]
    }
    const int recv = total;
    if (tid == 0) excl[F] = recv;
    __syncthreads();
    // Er + 1 entries: one more than the block's threads when Er = blockDim.x
    for (int j = tid; j <= Er; j += blockDim.x) grp_off[(size_t)r * (Er + 1) + j] = excl[j * N];
    if (tid < Er) m_sizes[(size_t)r * Er + tid] = excl[(tid + 1) * N] - excl[tid * N];
    if (tid == 0 && recv > cap) flag(status, MOE_ST_CAPACITY);
    const int wi = block_inclusive_scan(w, wsum, &total);
    if (tid < N) csend_off[(size_t)r * (N + 1) + tid] = wi - w;
    if (tid == 0) csend_off[(size_t)r * (N + 1) + N] = total;
}

__global__ void __launch_bounds__(1024)
    k_exchange(int N, int E, int cap, const int32_t *__restrict__ cnt,
               const int32_t *__restrict__ send_off, int32_t *__restrict__ grp_off,
               int32_t *__restrict__ seg_off, int32_t *__restrict__ csend_off,
               int32_t *__restrict__ m_sizes, int32_t *__restrict__ status) {
    const int r = blockIdx.x, tid = threadIdx.x, Er = E / N, F = Er * N;
    // runs in (local expert j, sender s) order: f = j*N + s
    const int j = tid / N, s = tid - (tid / N) * N;
    const int v = tid < F ? __ldg(cnt + (size_t)s * E + r * Er + j) : 0;
    // rows going back to each sender, in sender order
    const int w = tid < N ? __ldg(send_off + (size_t)tid * (N + 1) + r + 1) -
                                __ldg(send_off + (size_t)tid * (N + 1) + r)
                          : 0;
    route_receiver(N, E, cap, v, w, grp_off, seg_off, csend_off, m_sizes, status);
}

// Rank that owns flat assignment index i.
__device__ __forceinline__ int sender_of(long long i, long long TR) {
    return (int)div_nonneg(i, TR);
}

// Both roles in one launch: block r is sender r (as k_route_count) and
// receiver r.  The receiver needs every sender's count for its own Er
// experts; rather than waiting for the other blocks it recounts them from all
// ranks' ids (N*T*R ints, read from L2), so no block waits on another.
__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route(int N, int T, int E, int R, int cap, const int32_t *__restrict__ idx,
            int32_t *__restrict__ cnt_out, int32_t *__restrict__ send_off,
            int32_t *__restrict__ eso_out, int32_t *__restrict__ slot_row,
            int32_t *__restrict__ grp_off, int32_t *__restrict__ seg_off,
            int32_t *__restrict__ csend_off, int32_t *__restrict__ m_sizes,
            int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    const int r = blockIdx.x, tid = threadIdx.x, Er = E / N, F = Er * N;
    int *rc = smem;  // [N][Er] counts of (sender, local expert), then reused
    for (int i = tid; i < F; i += blockDim.x) rc[i] = 0;
    __syncthreads();
    const long long all = (long long)N * T * R, TR = (long long)T * R;
    const int lo = r * Er;
    // four ids per 16-byte load, four loads in flight per thread
    const long long n4 = all >> 2;
    const int4 *id4 = reinterpret_cast<const int4 *>(idx);
    for (long long i0 = tid; i0 < n4; i0 += 4LL * blockDim.x) {
        int4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long i = i0 + (long long)u * blockDim.x;
            v[u] = i < n4 ? __ldg(id4 + i) : make_int4(-1, -1, -1, -1);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long i = (i0 + (long long)u * blockDim.x) * 4;
            const int e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const unsigned j = (unsigned)(e4[q] - lo);
                // only 1 in N ids land here: the sender's index is worked out then
                if (j < (unsigned)Er) atomicAdd(&rc[sender_of(i + q, TR) * Er + (int)j], 1);
            }
        }
    }
    for (long long i = (n4 << 2) + tid; i < all; i += blockDim.x) {
        const unsigned j = (unsigned)(__ldg(idx + i) - lo);
        if (j < (unsigned)Er) atomicAdd(&rc[sender_of(i, TR) * Er + (int)j], 1);
    }
    __syncthreads();
    int v = 0, w = 0;
    if (tid < F) {
        const int j = tid / N, s = tid - j * N;
        v = rc[s * Er + j];
    }
    if (tid < N)
        for (int j = 0; j < Er; ++j) w += rc[tid * Er + j];
    route_receiver(N, E, cap, v, w, grp_off, seg_off, csend_off, m_sizes, status);
    if (route_sender(N, T, E, R, idx, cnt_out, send_off, eso_out, slot_row, smem) &&
        threadIdx.x == 0)
        flag(status, MOE_ST_BAD_EXPERT);
}

cudaError_t launch_route_count(const moe_shape &sh, const int32_t *idx, int32_t *cnt,
                               int32_t *send_off, int32_t *eso, int32_t *slot_row,
                               int32_t *status, cudaStream_t st) {
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return err;
    const size_t smem = route_smem(sh.E);
    static LaunchMemo attr;  // room for the largest E, once per device
    int set = 0;
    err = attr.get(0, &set, [](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(k_route_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)route_smem(MOE_MAX_EXPERTS));
    });
    if (err != cudaSuccess) return err;
    k_route_count<<<sh.N, kRouteThreads, smem, st>>>(sh.N, sh.T, sh.E, sh.R, idx, cnt, send_off,
                                                     eso, slot_row, status);
    return cudaGetLastError();
}

// Both roles in one launch with every rank's block in one thread-block
// cluster: each block plays sender (its counts go to expert_count), all
// blocks meet at a cluster barrier (release / acquire at cluster scope), and
// each block then plays receiver, reading the other senders' counts back
// through L2 -- the routing-information exchange of the pages, between the
// SMs of one cluster.  Block 0 clears *status before the barrier and every
// status bit is raised after it, so no separate clear precedes the launch.
// kGrid: the same for more ranks than a cluster holds, as a cooperative
// launch (every block resident) meeting at a grid-wide barrier instead.
// MOE_ROUTE_DSMEM: in the cluster form, receivers read every sender's
// scanned counts from the sender block's shared memory (one cluster barrier,
// the outputs written afterwards) instead of through L2 after the outputs;
// on the DSv3 EP16 route it measured 12.2 us against 11.3 us.
#ifndef MOE_ROUTE_DSMEM
#define MOE_ROUTE_DSMEM 0
#endif
#ifndef MOE_ROUTE_TRIGGER
#define MOE_ROUTE_TRIGGER 1
#endif

template <bool kGrid>
__global__ void __launch_bounds__(kRouteThreads, 1)
    k_route_cluster(int N, int T, int E, int R, int cap, const int32_t *__restrict__ idx,
                    int32_t *__restrict__ cnt_out, int32_t *__restrict__ send_off,
                    int32_t *__restrict__ eso_out, int32_t *__restrict__ slot_row,
                    int32_t *__restrict__ grp_off, int32_t *__restrict__ seg_off,
                    int32_t *__restrict__ csend_off, int32_t *__restrict__ m_sizes,
                    int32_t *__restrict__ status) {
    extern __shared__ int smem[];
    // a kernel launched after this one as its programmatic dependent may start
    // now (it waits on the device for this kernel's outputs)
    if (MOE_ROUTE_TRIGGER) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0;
    int rk[kAhead];
    SenderShare sh;
    const bool bad = sender_count<true, MOE_ROUTE_REG_RANKS>(N, T, E, R, blockIdx.x, idx, slot_row, smem, rk, sh);
    const int r = blockIdx.x, tid = threadIdx.x, Er = E / N, F = Er * N;
    const int j = tid / N, s = tid - (tid / N) * N;
    int v = 0, w = 0;
    constexpr bool kDsmem = !kGrid && MOE_ROUTE_DSMEM;
    if constexpr (!kDsmem) {
        // every sender output first, then the barrier (grid-wide, or the
        // cluster's), then each receiver reads the counts back through L2
        sender_write(N, T, E, R, idx, cnt_out, send_off, eso_out, slot_row, smem, rk, sh, true,
                     true);
        if constexpr (kGrid) {
            cooperative_groups::this_grid().sync();
        } else {
            asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        }
        // written by other blocks in this launch: read through L2, not the read-only path
        if (tid < F) v = __ldcg(cnt_out + (size_t)s * E + r * Er + j);
        if (tid < N)
            w = __ldcg(send_off + (size_t)tid * (N + 1) + r + 1) -
                __ldcg(send_off + (size_t)tid * (N + 1) + r);
    } else {
        // every sender's scanned counts straight from its block's shared
        // memory (distributed shared memory of the cluster; block s is
        // cluster rank s), after one cluster barrier
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (tid < F) {
            const uint32_t b = dsmem_addr(smem + r * Er + j, s);
            v = ld_dsmem(b + 4) - ld_dsmem(b);
        }
        if (tid < N) {
            const uint32_t b = dsmem_addr(smem, tid);
            w = ld_dsmem(b + 4u * (uint32_t)((r + 1) * Er)) - ld_dsmem(b + 4u * (uint32_t)(r * Er));
        }
        // done with the other blocks' shared memory (waited for before exit)
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    }
    if (bad && tid == 0) flag(status, MOE_ST_BAD_EXPERT);
    route_receiver(N, E, cap, v, w, grp_off, seg_off, csend_off, m_sizes, status);
    if constexpr (kDsmem) {
        sender_write(N, T, E, R, idx, cnt_out, send_off, eso_out, slot_row, smem, rk, sh, true,
                     true);
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    }
}

// Largest cluster k_route_cluster can be launched with on this device for E
// experts (0: none).
static int route_cluster_limit(int E) {
    static LaunchMemo memo;
    int limit = 0;
    const cudaError_t err = memo.get(E, &limit, [&](int *v) {
        *v = 0;
        if (cudaFuncSetAttribute(k_route_cluster<false>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
            cudaFuncSetAttribute(k_route_cluster<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)route_smem(MOE_MAX_EXPERTS)) != cudaSuccess) {
            cudaGetLastError();
            return cudaSuccess;
        }
        for (int c = 16; c >= 2; c >>= 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(c);
            cfg.blockDim = dim3(kRouteThreads);
            cfg.dynamicSmemBytes = route_smem(E);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k_route_cluster<false>, &cfg) == cudaSuccess &&
                n >= 1) {
                *v = c;
                break;
            }
            cudaGetLastError();
        }
        return cudaSuccess;
    });
    return err == cudaSuccess ? limit : 0;
}

// Most ranks whose route blocks can all be resident at once (0: none).
static int route_grid_limit(int E) {
    static LaunchMemo memo;
    int limit = 0;
    const cudaError_t err = memo.get(E, &limit, [&](int *v) {
        int occ = 0;
        *v = 0;
        if (cudaFuncSetAttribute(k_route_cluster<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)route_smem(MOE_MAX_EXPERTS)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_route_cluster<true>,
                                                          kRouteThreads,
                                                          route_smem(E)) != cudaSuccess) {
            cudaGetLastError();
            return cudaSuccess;
        }
        *v = occ * sm_count();
        return cudaSuccess;
    });
    return err == cudaSuccess ? limit : 0;
}

cudaError_t launch_route(const moe_shape &sh, int cap, const int32_t *idx, int32_t *cnt,
                         int32_t *send_off, int32_t *eso, int32_t *slot_row, int32_t *grp_off,
                         int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes, int32_t *status,
                         cudaStream_t st) {
    static LaunchMemo attr;
    int set = 0;
    cudaError_t err = attr.get(0, &set, [](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)route_smem(MOE_MAX_EXPERTS));
    });
    if (err != cudaSuccess) return err;
    if (sh.N > 1 && sh.N <= route_cluster_limit(sh.E)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(sh.N);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = route_smem(sh.E);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = sh.N;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // the kernel clears *status itself
        return cudaLaunchKernelEx(&cfg, k_route_cluster<false>, sh.N, sh.T, sh.E, sh.R, cap, idx,
                                  cnt, send_off, eso, slot_row, grp_off, seg_off, csend_off,
                                  m_sizes, status);
    }
    if (sh.N > 1 && sh.N <= route_grid_limit(sh.E))  // clears *status itself too
        return launch_kernel_coresident(k_route_cluster<true>, dim3(sh.N), dim3(kRouteThreads),
                                        route_smem(sh.E), st, sh.N, sh.T, sh.E, sh.R, cap, idx,
                                        cnt, send_off, eso, slot_row, grp_off, seg_off,
                                        csend_off, m_sizes, status);
    err = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return err;
    k_route<<<sh.N, kRouteThreads, route_smem(sh.E), st>>>(sh.N, sh.T, sh.E, sh.R, cap, idx, cnt,
                                                         send_off, eso, slot_row, grp_off, seg_off,
                                                         csend_off, m_sizes, status);
    return cudaGetLastError();
}

cudaError_t launch_exchange(const moe_shape &sh, int cap, const int32_t *cnt,
                            const int32_t *send_off, int32_t *grp_off, int32_t *seg_off,
                            int32_t *csend_off, int32_t *m_sizes, int32_t *status,
                            cudaStream_t st) {
    k_exchange<<<sh.N, 1024, 0, st>>>(sh.N, sh.E, cap, cnt, send_off, grp_off, seg_off, csend_off,
                                      m_sizes, status);
    return cudaGetLastError();
}

}  // namespace moe
