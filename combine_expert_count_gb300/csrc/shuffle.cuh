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

template <int U, class Map>
__global__ void __launch_bounds__(256)
    k_row_copy(const Map m, long long row0, long long nrows, long long rows_per_warp) {
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long r0 = gw * rows_per_warp;
    const long long r1 = min(nrows, r0 + rows_per_warp);
    const int nA = m.vecs_a(), nB = m.vecs_b();

    for (long long b = r0; b < r1; b += 32) {
        RowIdx d = {0, 0, 0};
        if (b + lane < r1) d = m.index(row0 + b + lane);
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
                    if (i < nA) v[u] = __ldcs(sa + i);
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
                for (int i = lane; i < nB; i += 32) db[i] = __ldcs(sb + i);
            }
        }
    }
}

}  // namespace moe
