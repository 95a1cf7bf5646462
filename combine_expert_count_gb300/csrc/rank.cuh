// rank.cuh -- the sender's counting pass shared by the routing kernels and
// the low-latency dispatch: per-expert counts of one rank's ids, their
// exclusive scan, and each id's rank among the equal ids of its warp's share
// ("Enabling trillion-parameter models on AWS EFA", section "Dispatch and
// combine": count per expert in one block, then a cumulative sum).
#pragma once

#include "common.cuh"

namespace moe {

// Rounds of 32 ids a warp loads before ranking any of them: a long share
// waits on one memory round trip per kAhead rounds, not per round.
constexpr int kAhead = 8;

// The lanes whose key equals this lane's, over the full warp (what
// __match_any_sync returns), for keys in [0, 2^nbits): one ballot per key
// bit, each lane keeping the lanes that agree with it on every bit.
#ifndef MOE_BALLOT_PEERS
#define MOE_BALLOT_PEERS 1
#endif
__device__ __forceinline__ unsigned warp_peers(int key, int nbits) {
    if (!MOE_BALLOT_PEERS) return __match_any_sync(kFull, key);
    unsigned peers = kFull;
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (key >> b) & 1;
        const unsigned m = __ballot_sync(kFull, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// Bits of the ranking keys: experts 0..E-1, and E for an id outside [0, E).
__device__ __forceinline__ int key_bits(int E) { return 32 - __clz(E); }

// Where a sender's warp keeps the ranks of its share between the passes:
// in registers when the share is one load round (rk), else in slot_row.
struct SenderShare {
    int lo, hi;      // the warp's share of the rank's flat ids
    bool one_round;  // hi - lo <= 32 * kAhead
};

// Sender role of rank s, part 1: counts and send offsets in shared memory
// only (except the ranks of shares longer than one round, kept in
// slot_row[s]).  Any block size that is a multiple of 32 works.
// Returns (the same in every thread) whether an id was outside [0, E).
//
// Stable slots in three passes, whatever T*R is: (1) warp w walks its own
// contiguous share of the rank's ids, 32 at a time; lanes holding the same
// expert find each other (warp_peers), the group's first lane adds
// the group to the warp's running count of that expert (a table row of its
// own, so no block barrier is needed) and every lane keeps "running count
// before its group + its rank in the group" -- its rank among equal ids in
// the warp's share; (2) per expert, the warps' counts become an exclusive
// prefix over warps, and their sum the expert's count, whose exclusive scan
// gives the send offsets (base); (3, sender_write) each lane adds its
// expert's offset and its warp's prefix.  The result equals "expert offset +
// number of earlier assignments with the same expert".
// kOneChunk: E <= blockDim.x (the routing kernels' 1024-thread blocks), so the
// expert scan is one block scan.  kRegRanks: single-round shares keep their
// ranks in registers (else every rank goes through slot_row).
template <bool kOneChunk = false, bool kRegRanks = true>
__device__ __forceinline__ bool sender_count(int N, int T, int E, int R, int s,
                                             const int32_t *__restrict__ idx,
                                             int32_t *__restrict__ slot_row, int *smem,
                                             int (&rk)[kAhead], SenderShare &sh) {
    int *base = smem;         // [E+1] exclusive scan of counts, then the total
    int *tab = base + E + 1;  // [nw][E] warp counts, then their exclusive prefix over warps
    __shared__ int wsum[32];
    __shared__ int total;
    __syncthreads();  // callers may reuse shared memory around this

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int TR = T * R;
    // warps that take ids (and own a table row): enough for 32 ids each, so a
    // short batch clears and sums few rows (one token per rank on 256
    // experts: the route took 8.9 us instead of 10.9 with all 32 warps)
    const int nw = max(1, min((int)(blockDim.x >> 5), TR / 32 + (TR % 32 != 0)));
    const int32_t *id = idx + (size_t)s * TR;
    int32_t *srow = slot_row + (size_t)s * TR;

    for (int i = tid; i < nw * E; i += blockDim.x) tab[i] = 0;
    __syncthreads();

    // 1. each warp's share: rank among equal ids, running counts per expert
    const int per = (TR + nw - 1) / nw;
    sh.lo = min(TR, warp * per);
    sh.hi = min(TR, sh.lo + per);
    sh.one_round = kRegRanks && sh.hi - sh.lo <= 32 * kAhead;
    const int lo = sh.lo, hi = sh.hi;
    int *mytab = tab + warp * E;
    const unsigned lt = (1u << lane) - 1u;
    const int nbits = key_bits(E);
    int bad = 0;
    for (int r0 = lo; r0 < hi; r0 += 32 * kAhead) {
        int ev[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int i = r0 + u * 32 + lane;
            ev[u] = i < hi ? __ldg(id + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            if (r0 + u * 32 >= hi) break;  // the same for the whole warp
            const int i = r0 + u * 32 + lane;
            const int e = ev[u];
            const bool good = (unsigned)e < (unsigned)E;
            if (i < hi && !good) bad = 1;
            const unsigned peers = warp_peers(good ? e : E, nbits);
            const int leader = __ffs(peers) - 1;
            int before = 0;
            if (good && lane == leader) {
                before = mytab[e];
                mytab[e] = before + __popc(peers);
            }
            before = __shfl_sync(kFull, before, leader);
            const int rank = good ? before + __popc(peers & lt) : -1;
            if (sh.one_round)
                rk[u] = rank;
            else if (i < hi)
                srow[i] = rank;
            __syncwarp();
        }
    }
    const bool any_bad = __syncthreads_or(bad) != 0;

    // 2. counts, prefix over warps, exclusive scan over experts (blockDim.x
    // experts at a time)
    if constexpr (kOneChunk) {
        int v = 0;
        if (tid < E) {
            for (int w = 0; w < nw; ++w) {
                const int c = tab[w * E + tid];
                tab[w * E + tid] = v;
                v += c;
            }
        }
        const int incl = block_inclusive_scan(v, wsum, &total);
        if (tid < E) base[tid] = incl - v;
        if (tid == 0) base[E] = total;
        __syncthreads();
        return any_bad;
    }
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + tid;
        int v = 0;
        if (e < E) {
            for (int w = 0; w < nw; ++w) {
                const int c = tab[w * E + e];
                tab[w * E + e] = v;
                v += c;
            }
        }
        const int incl = block_inclusive_scan(v, wsum, &total);
        if (e < E) base[e] = carry + incl - v;
        carry += total;
        __syncthreads();  // every thread has read `total` before the next scan
    }
    if (tid == 0) base[E] = carry;
    __syncthreads();
    return any_bad;
}

// Pass 3 of the sender: for every id of the warp's share, in order,
// put(i, e, u) with i its flat index in the rank, e its expert (ids outside
// [0, E) get e = -1) and u = the number of earlier ids of the rank with the
// same expert (the warp's exclusive prefix plus the rank within the warp).
template <class Put>
__device__ __forceinline__ void sender_ranks(int T, int E, int R, int s,
                                             const int32_t *__restrict__ idx,
                                             const int32_t *__restrict__ slot_row,
                                             const int *smem, const int (&rk)[kAhead],
                                             const SenderShare &sh, Put &&put) {
    const int *tab = smem + E + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, TR = T * R;
    const int32_t *id = idx + (size_t)s * TR;
    const int32_t *srow = slot_row + (size_t)s * TR;
    for (int r0 = sh.lo; r0 < sh.hi; r0 += 32 * kAhead) {
        int ev[kAhead], rv[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int i = r0 + u * 32 + lane;
            ev[u] = -1;
            rv[u] = 0;
            if (i < sh.hi) {
                ev[u] = __ldg(id + i);
                rv[u] = sh.one_round ? rk[u] : srow[i];  // this lane's own pass-1 rank
            }
        }
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int i = r0 + u * 32 + lane;
            const int e = ev[u];
            if (i < sh.hi) {
                const bool good = (unsigned)e < (unsigned)E;
                put(i, good ? e : -1, good ? tab[warp * E + e] + rv[u] : 0);
            }
        }
    }
}

}  // namespace moe
