// shuffle.cuh -- row-permuting copy used by the dispatch receive shuffle and
// the combine send pack.
//
// Work is the flat list of send-buffer rows (s, i), s < N, i < T*R; every
// row has exactly one destination.  Each warp owns a contiguous range of
// rows.  For a batch of 32 rows the lanes work out, in parallel, where each
// row goes (Map::index: pure index arithmetic on the routing arrays) and
// write the row's side data (Map::side); then the warp moves the rows one by
// one, 16-byte vectors, U per lane in flight.  Occupancy (many warps per SM)
// supplies the bytes in flight.
//
// A measured alternative -- one warp per CTA streaming rows through a
// shared-memory ring with cp.async.bulk loads and stores -- was slower on
// GB300 (one issuing thread per CTA limits the copies in flight).
#pragma once

#include "common.cuh"

namespace moe {

struct RowIdx {
    int kind;       // 0: nothing to move, 1: copy, 2: write zeros to the destination
    long long src;  // source row (map units)
    long long dst;  // destination row
};

// Rows [r0, r1) of the flat list (offset by row0), by one warp.  A Map with
// kWaits == true makes each row wait (Map::ready, bounded by one cycle budget
// for the whole warp) until its source rows have been published; Map::ld is
// the load used for the payload.
template <int U, class Map>
__device__ __forceinline__ void copy_rows(const Map &m, long long row0, long long r0,
                                          long long r1) {
    const int lane = threadIdx.x & 31;
    const int nA = m.vecs_a(), nB = m.vecs_b();
    long long deadline = 0;
    if constexpr (Map::kWaits) deadline = clock64() + kWaitCycles;

    for (long long b = r0; b < r1; b += 32) {
        RowIdx d = {0, 0, 0};
        if (b + lane < r1) d = m.index(row0 + b + lane);
        if constexpr (Map::kWaits) {
            m.ready(d, deadline);
            // lane q acquired row q's flag, but every lane reads row q: the
            // warp barrier orders that acquire before the other lanes' loads
            __syncwarp();
        }
        if (d.kind == 1) m.side(d);
        const int cnt = (int)min(32LL, r1 - b);
        for (int q = 0; q < cnt; ++q) {
            const int kind = __shfl_sync(kFull, d.kind, q);
            if (kind == 0) continue;
            const long long dst = __shfl_sync(kFull, d.dst, q);
            uint4 *da = m.dst_a(dst);
            if (kind == 2) {
                for (int i = lane; i < nA; i += 32) da[i] = make_uint4(0, 0, 0, 0);
                continue;
            }
            const long long src = __shfl_sync(kFull, d.src, q);
            const uint4 *sa = m.src_a(src);
            for (int i0 = 0; i0 < nA; i0 += 32 * U) {
                uint4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = i0 + u * 32 + lane;
                    if (i < nA) v[u] = m.ld(sa + i);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = i0 + u * 32 + lane;
                    if (i < nA) da[i] = v[u];
                }
            }
            if (nB) {
                const uint4 *sb = m.src_b(src);
                uint4 *db = m.dst_b(dst);
                for (int i = lane; i < nB; i += 32) db[i] = m.ld(sb + i);
            }
        }
    }
}

template <int U, class Map>
__global__ void __launch_bounds__(256)
    k_row_copy(const Map m, long long row0, long long nrows, long long rows_per_warp) {
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long r0 = gw * rows_per_warp;
    const long long r1 = min(nrows, r0 + rows_per_warp);
    copy_rows<U, Map>(m, row0, r0, r1);
}

// Row i of sender s belongs to expert e (the run of expert_send_off[s] that
// holds i), hosted by r = e/Er as local expert j; it lands at grouped row
// seg_off[r][j][s] + (i - expert_send_off[s][e]).  Shared by both maps.
struct RowRoute {
    int s, i, r, g;
    bool valid;
};

__device__ __forceinline__ RowRoute route_row(long long f, long long TR, int N, int E, int Er,
                                              const int32_t *__restrict__ eso,
                                              const int32_t *__restrict__ seg_off) {
    RowRoute rr;
    rr.s = (int)div_nonneg(f, TR);
    rr.i = (int)(f - (long long)rr.s * TR);
    const int32_t *es = eso + (size_t)rr.s * (E + 1);
    rr.valid = rr.i < __ldg(es + E);  // beyond the rows s packed: nothing
    rr.r = 0;
    rr.g = 0;
    if (!rr.valid) return rr;
    const int e = find_run(es, E, rr.i);
    rr.r = e / Er;
    const int j = e - rr.r * Er;
    rr.g = __ldg(seg_off + ((size_t)rr.r * Er + j) * N + rr.s) + (rr.i - __ldg(es + e));
    return rr;
}

// The dispatch receive: send row (s, i) -> grouped row of rank r.
// kWait: the send rows are written by other CTAs of the same kernel, which
// publish each (sender s, receiver r) group with published[s][r] = 1; a row is
// copied only once its group is published, and every read of what those
// CTAs wrote goes to L2 (never the non-coherent or L1 paths).
template <bool kWait>
struct DispatchMapT {
    static constexpr bool kWaits = kWait;
    int N, E, Er, Sb, cap, H;
    long long TR;
    bool bulk_scales;  // scale rows are whole 16-byte vectors: move them with the payload
    const uint8_t *send_q;
    const float *send_s;
    const int32_t *send_tok, *eso, *seg_off;
    uint8_t *grp_q;
    float *grp_s;
    int32_t *grp_src;
    const int32_t *published;  // kWait: [N][N] group flags, 1 once written
    int32_t *status;       // kWait: MOE_ST_TIMEOUT when a group never appears

    __device__ __forceinline__ int vecs_a() const { return H >> 4; }
    __device__ __forceinline__ int vecs_b() const { return bulk_scales ? Sb >> 2 : 0; }

    template <class V>
    __device__ __forceinline__ V ld(const V *p) const {
        if constexpr (kWait)
            return __ldcg(p);
        else
            return __ldcs(p);
    }

    __device__ __forceinline__ RowIdx index(long long f) const {
        const RowRoute rr = route_row(f, TR, N, E, Er, eso, seg_off);
        RowIdx d = {0, 0, 0};
        // a grouped row at or past cap is dropped (the exchange flagged it)
        if (!rr.valid || rr.g < 0 || rr.g >= cap) return d;
        d.kind = 1;
        d.src = (long long)rr.s * TR + rr.i;
        d.dst = (long long)rr.r * cap + rr.g;
        return d;
    }
    // Bounded wait for the row's (s, r) group; on timeout the row is skipped.
    __device__ __forceinline__ void ready_wait(RowIdx &d, long long deadline) const {
        if (d.kind != 1) return;
        const int s = (int)div_nonneg(d.src, TR), r = (int)div_nonneg(d.dst, cap);
        const int32_t *f = published + (size_t)s * N + r;
        while (ld_acquire(f) == 0) {
            if (clock64() > deadline) {
                flag(status, MOE_ST_TIMEOUT);
                d.kind = 0;
                return;
            }
            __nanosleep(256);
        }
    }
    __device__ __forceinline__ void ready(RowIdx &d, long long deadline) const {
        if constexpr (kWait) ready_wait(d, deadline);
    }
    __device__ __forceinline__ void side(const RowIdx &d) const {
        const int s = (int)div_nonneg(d.src, TR);
        const int tok = kWait ? __ldcg(send_tok + d.src) : __ldg(send_tok + d.src);
        *reinterpret_cast<int2 *>(grp_src + d.dst * 2) = make_int2(s, tok);
        if (!bulk_scales)
            for (int b = 0; b < Sb; ++b)
                grp_s[d.dst * Sb + b] = kWait ? __ldcg(send_s + d.src * Sb + b)
                                              : __ldg(send_s + d.src * Sb + b);
    }
    __device__ __forceinline__ const uint4 *src_a(long long row) const {
        return reinterpret_cast<const uint4 *>(send_q + row * H);
    }
    __device__ __forceinline__ uint4 *dst_a(long long row) const {
        return reinterpret_cast<uint4 *>(grp_q + row * H);
    }
    __device__ __forceinline__ const uint4 *src_b(long long row) const {
        return reinterpret_cast<const uint4 *>(send_s + row * Sb);
    }
    __device__ __forceinline__ uint4 *dst_b(long long row) const {
        return reinterpret_cast<uint4 *>(grp_s + row * Sb);
    }
};

using DispatchMap = DispatchMapT<false>;

}  // namespace moe
