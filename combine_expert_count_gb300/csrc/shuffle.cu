// shuffle.cu -- the two row shuffles of the path, both driven by the
// bulk-copy pipeline in shuffle.cuh:
//   dispatch receive: send buffers -> expert-grouped layout for the grouped
//     GEMM ("Enabling trillion-parameter models on AWS EFA", section
//     "Dispatch and combine": received tokens are shuffled into the tensor
//     passed to the grouped GEMM);
//   combine send: expert outputs -> per-destination contiguous combine send
//     buffers ("one write per peer").
// The N ranks are slices of one GPU, so the wire is the pull itself: the
// receiving side reads the sender's slice directly.
#include "common.cuh"
#include "launch.h"
#include "shuffle.cuh"

namespace moe {

constexpr int kDispStages = 6, kDispDepth = 4;

// ------------------------------------------------------------ receive shuffle
//
// Row i of sender s belongs to expert e (the run of expert_send_off[s] that
// holds i), hosted by r = e/Er as local expert j; it lands at grouped row
// seg_off[r][j][s] + (i - expert_send_off[s][e]).
struct DispatchMap {
    int N, E, Er, Sb, cap, H;
    long long TR;
    bool bulk_scales;
    const uint8_t *send_q;
    const float *send_s;
    const int32_t *send_tok, *eso, *seg_off;
    uint8_t *grp_q;
    float *grp_s;
    int32_t *grp_src;

    __device__ __forceinline__ RowDesc map(long long f) const {
        RowDesc d;
        d.kind = 0;
        const int s = (int)(f / TR);
        const int i = (int)(f - (long long)s * TR);
        const int32_t *es = eso + (size_t)s * (E + 1);
        if (i >= __ldg(es + E)) return d;  // beyond the rows s packed
        const int e = find_run(es, E, i);
        const int r = e / Er, j = e - r * Er;
        const int g = __ldg(seg_off + ((size_t)r * Er + j) * N + s) + (i - __ldg(es + e));
        if (g < 0 || g >= cap) return d;  // dropped: the exchange flagged MOE_ST_CAPACITY
        const size_t srow = (size_t)s * TR + i, drow = (size_t)r * cap + g;
        d.kind = 1;
        d.srcA = reinterpret_cast<const char *>(send_q + srow * H);
        d.dstA = reinterpret_cast<char *>(grp_q + drow * H);
        if (bulk_scales) {
            d.srcB = reinterpret_cast<const char *>(send_s + srow * Sb);
            d.dstB = reinterpret_cast<char *>(grp_s + drow * Sb);
        } else {
            d.srcB = nullptr;
            d.dstB = nullptr;
            for (int b = 0; b < Sb; ++b) grp_s[drow * Sb + b] = __ldg(send_s + srow * Sb + b);
        }
        *reinterpret_cast<int2 *>(grp_src + drow * 2) = make_int2(s, __ldg(send_tok + srow));
        return d;
    }
};

template <int S, int L, class Map>
static cudaError_t launch_shuffle(const Map &m, const ShuffleGeom &g, long long nrows,
                                  int32_t *status, cudaStream_t st) {
    if (nrows == 0) return cudaSuccess;
    auto kern = k_row_shuffle<S, L, Map>;
    // + 128: the kernel aligns the stage base itself
    const int smem = (int)(S * g.stage_bytes + 128);
    static int cached_dev = -1, cached_smem = -1, cached_occ = 1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev != cached_dev || smem != cached_smem) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        int occ = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32, smem);
        if (err != cudaSuccess) return err;
        cached_occ = occ < 1 ? 1 : occ;
        cached_dev = dev;
        cached_smem = smem;
    }
    const int occ = cached_occ;
    long long grid = (long long)sm_count() * occ;
    if (grid > nrows) grid = nrows;
    const long long per = (nrows + grid - 1) / grid;
    grid = (nrows + per - 1) / per;
    kern<<<(int)grid, 32, smem, st>>>(m, g, nrows, per, status);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_pull(const moe_shape &sh, int cap, const uint8_t *send_q,
                                 const float *send_s, const int32_t *send_tok,
                                 const int32_t *eso, const int32_t *seg_off, uint8_t *grp_q,
                                 float *grp_s, int32_t *grp_src, int32_t *status,
                                 cudaStream_t st) {
    DispatchMap m;
    m.N = sh.N;
    m.E = sh.E;
    m.Er = sh.E / sh.N;
    m.Sb = sh.H / 128;
    m.cap = cap;
    m.H = sh.H;
    m.TR = (long long)sh.T * sh.R;
    m.bulk_scales = (m.Sb % 4) == 0;  // scale rows are whole 16-byte units
    m.send_q = send_q;
    m.send_s = send_s;
    m.send_tok = send_tok;
    m.eso = eso;
    m.seg_off = seg_off;
    m.grp_q = grp_q;
    m.grp_s = grp_s;
    m.grp_src = grp_src;
    const ShuffleGeom g = make_geom((uint32_t)sh.H, m.bulk_scales ? (uint32_t)(m.Sb * 4) : 0u);
    return launch_shuffle<kDispStages, kDispDepth>(m, g, (long long)sh.N * m.TR, status, st);
}

// ------------------------------------------------------------ combine pack
//
// The same row (s, i) as above, now for the way back: expert rank r copies
// its output row (grouped row g) to its combine send buffer at
// csend_off[r][s] + (i - send_off[s][r]), the position row i has inside the
// run s sent to r.  If g was dropped for capacity the row is sent as zeros.
struct CombineMap {
    int N, E, Er, cap, H;
    long long TR;
    const uint16_t *y;
    const int32_t *eso, *send_off, *seg_off, *csend_off;
    uint16_t *csend;

    __device__ __forceinline__ RowDesc map(long long f) const {
        RowDesc d;
        d.kind = 0;
        d.srcB = nullptr;
        d.dstB = nullptr;
        const int s = (int)(f / TR);
        const int i = (int)(f - (long long)s * TR);
        const int32_t *es = eso + (size_t)s * (E + 1);
        if (i >= __ldg(es + E)) return d;
        const int e = find_run(es, E, i);
        const int r = e / Er, j = e - r * Er;
        const int g = __ldg(seg_off + ((size_t)r * Er + j) * N + s) + (i - __ldg(es + e));
        const int c = __ldg(csend_off + (size_t)r * (N + 1) + s) +
                      (i - __ldg(send_off + (size_t)s * (N + 1) + r));
        if (c < 0 || c >= cap) return d;
        d.dstA = reinterpret_cast<char *>(csend + ((size_t)r * cap + c) * H);
        if (g < 0 || g >= cap) {
            d.kind = 2;  // the expert never saw this row: send zeros
            return d;
        }
        d.kind = 1;
        d.srcA = reinterpret_cast<const char *>(y + ((size_t)r * cap + g) * H);
        return d;
    }
};

constexpr int kCombStages = 4, kCombDepth = 3;

cudaError_t launch_combine_pack(const moe_shape &sh, int cap, const uint16_t *y,
                                const int32_t *eso, const int32_t *send_off,
                                const int32_t *seg_off, const int32_t *csend_off, uint16_t *csend,
                                int32_t *status, cudaStream_t st) {
    CombineMap m;
    m.N = sh.N;
    m.E = sh.E;
    m.Er = sh.E / sh.N;
    m.cap = cap;
    m.H = sh.H;
    m.TR = (long long)sh.T * sh.R;
    m.y = y;
    m.eso = eso;
    m.send_off = send_off;
    m.seg_off = seg_off;
    m.csend_off = csend_off;
    m.csend = csend;
    const ShuffleGeom g = make_geom((uint32_t)sh.H * 2u, 0u);
    return launch_shuffle<kCombStages, kCombDepth>(m, g, (long long)sh.N * m.TR, status, st);
}

}  // namespace moe
