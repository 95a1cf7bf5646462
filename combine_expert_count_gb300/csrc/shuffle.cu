// shuffle.cu -- the two row shuffles of the path, both driven by k_row_copy
// (the dispatch map and the row routing live in shuffle.cuh):
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

#ifndef MOE_DISP_VECS
#define MOE_DISP_VECS 14
#endif
#ifndef MOE_COMB_VECS
#define MOE_COMB_VECS 14
#endif

namespace moe {

// The same row (s, i), now for the way back: expert rank r copies its output
// row (grouped row g) to its combine send buffer at
// csend_off[r][s] + (i - send_off[s][r]), the position row i has inside the
// run s sent to r.  If g was dropped for capacity the row is sent as zeros.
struct CombineMap {
    static constexpr bool kWaits = false;
    int N, E, Er, cap, H;
    long long TR;
    const uint16_t *y;
    const int32_t *eso, *send_off, *seg_off, *csend_off;
    uint16_t *csend;

    __device__ __forceinline__ int vecs_a() const { return H >> 3; }
    __device__ __forceinline__ int vecs_b() const { return 0; }

    __device__ __forceinline__ RowIdx index(long long f) const {
        const RowRoute rr = route_row(f, TR, N, E, Er, eso, seg_off);
        RowIdx d = {0, 0, 0};
        if (!rr.valid) return d;
        const int c = __ldg(csend_off + (size_t)rr.r * (N + 1) + rr.s) +
                      (rr.i - __ldg(send_off + (size_t)rr.s * (N + 1) + rr.r));
        if (c < 0 || c >= cap) return d;
        d.dst = (long long)rr.r * cap + c;
        if (rr.g < 0 || rr.g >= cap) {
            d.kind = 2;  // the expert never saw this row: send zeros
            return d;
        }
        d.kind = 1;
        d.src = (long long)rr.r * cap + rr.g;
        return d;
    }
    __device__ __forceinline__ void ready(RowIdx &, long long) const {}
    __device__ __forceinline__ void side(const RowIdx &) const {}
    template <class V>
    __device__ __forceinline__ V ld(const V *p) const {
        return __ldcs(p);
    }
    __device__ __forceinline__ const uint4 *src_a(long long row) const {
        return reinterpret_cast<const uint4 *>(y + row * H);
    }
    __device__ __forceinline__ uint4 *dst_a(long long row) const {
        return reinterpret_cast<uint4 *>(csend + row * H);
    }
    __device__ __forceinline__ const uint4 *src_b(long long) const { return nullptr; }
    __device__ __forceinline__ uint4 *dst_b(long long) const { return nullptr; }
};

// 256-thread blocks, grid sized to residency, rows split evenly over warps.
template <int U, class Map>
static cudaError_t launch_copy(const Map &m, long long row0, long long nrows,
                               cudaStream_t st) {
    if (nrows <= 0) return cudaSuccess;
    auto kern = k_row_copy<U, Map>;
    static LaunchMemo memo;
    int occ = 1;
    cudaError_t err = memo.get(0, &occ, [&](int *v) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, 256, 0);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    long long warps = (long long)sm_count() * occ * 8;
    if (warps > nrows) warps = nrows;
    const long long per = (nrows + warps - 1) / warps;
    warps = (nrows + per - 1) / per;
    const long long grid = (warps + 7) / 8;
    return launch_kernel(kern, dim3((unsigned)grid), dim3(256), 0, st, m, row0, nrows, per);
}

cudaError_t launch_dispatch_pull(const moe_shape &sh, int cap, const uint8_t *send_q,
                                 const float *send_s, const int32_t *send_tok,
                                 const int32_t *eso, const int32_t *seg_off, uint8_t *grp_q,
                                 float *grp_s, int32_t *grp_src, int32_t *status,
                                 cudaStream_t st, long long row0, long long row1) {
    (void)status;
    DispatchMap m;
    m.N = sh.N;
    m.E = sh.E;
    m.Er = sh.E / sh.N;
    m.Sb = sh.H / 128;
    m.cap = cap;
    m.H = sh.H;
    m.TR = (long long)sh.T * sh.R;
    m.bulk_scales = (m.Sb % 4) == 0;
    m.send_q = send_q;
    m.send_s = send_s;
    m.send_tok = send_tok;
    m.eso = eso;
    m.seg_off = seg_off;
    m.grp_q = grp_q;
    m.grp_s = grp_s;
    m.grp_src = grp_src;
    m.published = nullptr;
    m.status = nullptr;
    if (row1 < 0) row1 = (long long)sh.N * m.TR;
    return launch_copy<MOE_DISP_VECS>(m, row0, row1 - row0, st);
}

cudaError_t launch_combine_pack(const moe_shape &sh, int cap, const uint16_t *y,
                                const int32_t *eso, const int32_t *send_off,
                                const int32_t *seg_off, const int32_t *csend_off, uint16_t *csend,
                                int32_t *status, cudaStream_t st, long long row0, long long row1) {
    (void)status;
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
    if (row1 < 0) row1 = (long long)sh.N * m.TR;
    return launch_copy<MOE_COMB_VECS>(m, row0, row1 - row0, st);
}

}  // namespace moe
