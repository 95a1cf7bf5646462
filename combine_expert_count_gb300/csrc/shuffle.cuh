// shuffle.cuh -- row-permuting copy through shared memory with bulk async
// copies (TMA, non-tensor form), used by the dispatch receive shuffle and the
// combine send pack.
//
// Work is the flat list of send-buffer rows (s, i), s < N, i < T*R; each CTA
// (one warp) owns a contiguous range of it.  For a batch of 32 rows the lanes
// compute where each row goes (Map::map, which also writes any per-row
// metadata); lane 0 then streams the rows through an S-stage ring in shared
// memory: a bulk load global->shared completes on the stage's mbarrier, a
// bulk store shared->global drains it.  Up to L loads are in flight; a stage
// is reloaded only once the store that last read it has finished reading
// (cp.async.bulk.wait_group.read), which with one commit group per row needs
// at most S-L younger groups pending.  Rows longer than kPiece bytes move in
// pieces.  Every mbarrier wait is bounded; on expiry the CTA stops issuing,
// raises MOE_ST_TIMEOUT and returns once its copies in flight are done.
#pragma once

#include "common.cuh"

namespace moe {

constexpr uint32_t kPiece = 16384;

struct RowDesc {
    int kind;  // 0: nothing to move, 1: copy A (+ B), 2: write zeros to dstA
    const char *srcA;
    char *dstA;
    const char *srcB;
    char *dstB;
};

struct ShuffleGeom {
    uint32_t bytesA;       // payload bytes per row (multiple of 16)
    uint32_t bytesB;       // side bytes per row moved in the same stage (0 or multiple of 16)
    uint32_t a_area;       // shared bytes reserved for one piece of A
    uint32_t stage_bytes;  // a_area + bytesB, rounded up to 128
};

inline ShuffleGeom make_geom(uint32_t bytesA, uint32_t bytesB) {
    ShuffleGeom g;
    g.bytesA = bytesA;
    g.bytesB = bytesB;
    g.a_area = bytesA < kPiece ? bytesA : kPiece;
    g.stage_bytes = (g.a_area + bytesB + 127u) & ~127u;
    return g;
}

template <int S>
struct Ring {
    uint64_t bar[S];
    char *dstA[S];
    char *dstB[S];
    uint32_t lenA[S];
    uint32_t lenB[S];
};

template <int S>
__device__ __forceinline__ bool ring_store(Ring<S> &ring, unsigned char *stage,
                                           const ShuffleGeom &g, long long n) {
    const int slot = (int)(n % S);
    if (!mbar_wait(&ring.bar[slot], (uint32_t)((n / S) & 1))) return false;
    unsigned char *sp = stage + (size_t)slot * g.stage_bytes;
    bulk_s2g(ring.dstA[slot], sp, ring.lenA[slot]);
    if (ring.lenB[slot]) bulk_s2g(ring.dstB[slot], sp + g.a_area, ring.lenB[slot]);
    bulk_commit();
    return true;
}

template <int S, int L, class Map>
__global__ void __launch_bounds__(32)
    k_row_shuffle(const Map m, const ShuffleGeom g, long long nrows, long long rows_per_cta,
                  int32_t *status) {
    static_assert(L >= 1 && L <= S, "pipeline depth");
    extern __shared__ __align__(128) unsigned char stage_raw[];
    // bulk copies need 16-byte aligned shared addresses: align the base to
    // 128 (the launch reserves the extra bytes)
    unsigned char *stage = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(stage_raw) + 127) & ~static_cast<uintptr_t>(127));
    __shared__ Ring<S> ring;
    __shared__ RowDesc desc[32];

    const int lane = threadIdx.x;
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&ring.bar[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const long long r0 = (long long)blockIdx.x * rows_per_cta;
    const long long r1 = min(nrows, r0 + rows_per_cta);
    long long nload = 0, nstore = 0;  // meaningful in lane 0 only
    bool ok = true;

    for (long long b = r0; b < r1; b += 32) {
        RowDesc d;
        d.kind = 0;
        if (b + lane < r1) d = m.map(b + lane);
        desc[lane] = d;
        __syncwarp();
        if (lane == 0) {
            for (int q = 0; q < 32 && ok; ++q) {
                const RowDesc dq = desc[q];
                if (dq.kind != 1) continue;
                for (uint32_t off = 0; off < g.bytesA && ok; off += kPiece) {
                    const uint32_t lenA = min(kPiece, g.bytesA - off);
                    const uint32_t lenB = off == 0 ? g.bytesB : 0u;
                    if (nload - nstore == L) {
                        if (!ring_store<S>(ring, stage, g, nstore)) {
                            ok = false;
                            break;
                        }
                        ++nstore;
                    }
                    const int slot = (int)(nload % S);
                    if (nload >= S) bulk_wait_read<S - L>();
                    unsigned char *sp = stage + (size_t)slot * g.stage_bytes;
                    mbar_arrive_expect_tx(&ring.bar[slot], lenA + lenB);
                    bulk_g2s(sp, dq.srcA + off, lenA, &ring.bar[slot]);
                    if (lenB) bulk_g2s(sp + g.a_area, dq.srcB, lenB, &ring.bar[slot]);
                    ring.dstA[slot] = dq.dstA + off;
                    ring.dstB[slot] = dq.dstB;
                    ring.lenA[slot] = lenA;
                    ring.lenB[slot] = lenB;
                    ++nload;
                }
            }
        }
        __syncwarp();
        for (int q = 0; q < 32; ++q) {
            if (desc[q].kind != 2) continue;
            uint4 *p = reinterpret_cast<uint4 *>(desc[q].dstA);
            for (uint32_t o = lane; o < g.bytesA / 16; o += 32) p[o] = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
    }

    if (lane == 0) {
        while (ok && nstore < nload) {
            if (!ring_store<S>(ring, stage, g, nstore)) {
                ok = false;
                break;
            }
            ++nstore;
        }
        bulk_wait_all();
        if (!ok) {
            flag(status, MOE_ST_TIMEOUT);
            // let the loads still in flight land before the CTA's shared memory goes away
            for (long long n = nstore; n < nload; ++n)
                mbar_wait(&ring.bar[n % S], (uint32_t)((n / S) & 1));
        }
    }
}

}  // namespace moe
