// dispatch.cu -- dispatch send: block-scaled fp8 quantisation fused with the
// pack into contiguous per-peer send buffers, after "Enabling
// trillion-parameter models on AWS EFA", sections "Dispatch and combine"
// (pack once the offsets are known) and "Evaluation: dispatch/combine
// latency" (block-scaled fp8 dispatch).
#include <cuda_fp8.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "rank.cuh"
#include "shuffle.cuh"

namespace moe {

// The conversion: two fp32 values to two e4m3 bytes (first value in the
// low byte), round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t cvt_pair(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// ------------------------------------------------------------ quant + pack
//
// One CTA works through (token, piece) items, a piece being up to
// kPieceElems elements of the row (a multiple of 128, so no scale block
// straddles two pieces).  Per item: the bf16 piece arrives in shared memory
// by one bulk copy (issued into a ring of x buffers up to kNB - 1 items
// ahead, completion on the buffer's mbarrier); the
// threads quantise it, 16 elements per thread and 8 threads per 128-element
// block (amax by xor-shuffles within the group, scale = amax/448 and
// q = e4m3_satfinite_rn(x/scale) with IEEE fp32 divisions), and each thread
// stores its 16 fp8 bytes straight from registers to the same place in each
// of the token's R destination rows (one 512-byte coalesced store per warp
// and row), the group's first thread also the scale.  The ring (four
// buffers for the send and fused forms, two for the others: x_stages) lets
// the loads of the next items overlap the arithmetic and stores of item n.
// The fused
// and low-latency forms store their fp8 rows evict-first (st.global.cs):
// nothing in the dispatch + combine step reads them again (the send rows are
// the wire copy; the grouped rows are read by the grouped GEMM, which runs
// between the two halves and outside this library), and the DSv3 EP16 layer
// (dispatch, then combine, as one graph) took 137.6 us against 138.8 with
// default stores, the dispatch itself unchanged.  A caller whose GEMM runs
// right after the dispatch and could find the grouped rows in L2 gives up
// that chance with these stores.  The send-only form keeps default
// stores: its rows are read back next (by the receive pull, or by the
// signalled kernel's own copy phase), which evict-first stores made 4 and
// 1.2 us slower.
//
// Measured against staging the fp8 piece in shared memory and sending it
// with R bulk (TMA) stores per destination: the direct stores are 2 us
// faster on the DSv3 EP16 dispatch (the bulk stores' shared-memory reads
// had to finish before a buffer could be reused).
#ifndef MOE_PIECE_ELEMS
#define MOE_PIECE_ELEMS 8192
#endif
constexpr int kPieceElems = MOE_PIECE_ELEMS;
static_assert(kPieceElems % 128 == 0, "pieces hold whole scale blocks");

// x buffers of the staged body: the load of item n + kNB - 1 is issued when
// item n starts, so a CTA keeps up to kNB - 1 pieces in flight (kNB when it
// prefetches before a gate).  The pack into the send buffer (and, fused, the
// grouped layout) uses MOE_PACK_STAGES buffers; its pieces are whole rows
// (up to kPieceElems) for batches of more than MOE_PACK_LONG tokens per
// resident CTA, else rows halved to at most MOE_PACK_PIECE elements (more,
// smaller items for short batches, and five CTAs per SM instead of three).
// The low-latency forms and the signalled dispatch, which spend per-item
// work on finding or publishing rows, use two buffers of whole rows.
// Measured on the layer graphs against two whole-row buffers: DSv3 EP16
// (2.7 tokens per CTA) 136.5 us with four half-row buffers, 138.9 with four
// whole-row ones, 136.5 with two; Kimi-K2 EP32 (5.4 tokens per CTA) 259.4,
// 257.5, 261.1; prefill EP8 (43 tokens per CTA) 1975, 1933, 1977; the
// low-latency dispatch took 40.4 against 35.9 us with half rows (its
// per-item search runs twice per token).
#ifndef MOE_PACK_STAGES
#define MOE_PACK_STAGES 4
#endif
#ifndef MOE_PACK_PIECE
#define MOE_PACK_PIECE 4096
#endif
#ifndef MOE_PACK_LONG
#define MOE_PACK_LONG 4
#endif
static_assert(MOE_PACK_STAGES >= 2 && MOE_PACK_STAGES <= 8, "two to eight x buffers");
static_assert(MOE_PACK_PIECE % 128 == 0, "pieces hold whole scale blocks");

// Buffers and largest piece of each form of the staged body.
enum class Dest { kSend, kSendGrouped, kLowLatency, kLowLatencyRanked };
__host__ __device__ constexpr int x_stages(Dest d, bool signal) {
    return (d == Dest::kSend || d == Dest::kSendGrouped) && !signal ? MOE_PACK_STAGES : 2;
}
__host__ __device__ constexpr int piece_cap(Dest d, bool signal, bool long_batch = false) {
    return (d == Dest::kSend || d == Dest::kSendGrouped) && !signal && !long_batch
               ? MOE_PACK_PIECE
               : kPieceElems;
}

// Shared memory of the staged body for piece size P and kNB buffers: the
// bf16 x buffers; the low-latency histogram or counting tables follow.
__host__ __device__ constexpr size_t stage_bytes(int P, int nb) { return (size_t)nb * 2 * P; }

__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float scale) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float f0 = bf16_lo(w[2 * u]), f1 = bf16_hi(w[2 * u]);
        const float f2 = bf16_lo(w[2 * u + 1]), f3 = bf16_hi(w[2 * u + 1]);
        const uint32_t lo = cvt_pair(__fdiv_rn(f0, scale), __fdiv_rn(f1, scale));
        const uint32_t hi = cvt_pair(__fdiv_rn(f2, scale), __fdiv_rn(f3, scale));
        o[u] = lo | (hi << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float amax16(const uint4 &a, const uint4 &b) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float m = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[u])), fabsf(bf16_hi(w[u]))));
    return m;
}

// Where the quantised rows go (Dest above): the send buffer
// (moe_dispatch_send), the send buffer and the grouped layout (fused
// dispatch), or the low-latency layout (rows found per token by the CTA, or
// ranked per sender first: kLowLatencyRanked).

// Low-latency layout: receiver r keeps a T-row region per (local expert j,
// sender s); assignment (t, k) of s with expert e = r*Er + j takes row
// ((r*Er + j)*N + s)*T + u, u = its stable rank among s's assignments to e.
struct LLDest {
    int N, E;
    const int32_t *idx;
    int32_t *ll_row;    // [N][T][R] row of each assignment, -1: none
    int32_t *ll_count;  // [N][Er][N] assignments per region
};

// What the staged body does once both x buffers' first loads are issued and
// before it reads anything another kernel or phase writes: nothing, wait for
// the routing kernel (programmatic dependent launch), or rank every sender's
// ids into the low-latency rows and meet at a grid-wide barrier.
struct NoGate {
    static constexpr bool kPrefetch = false;
    __device__ __forceinline__ void operator()(int *) const {}
};

struct PdlGate {
    static constexpr bool kPrefetch = true;
    __device__ __forceinline__ void operator()(int *) const {
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
};

// Where the grouped copy of each assignment goes, for the fused dispatch:
// row i = slot of rank s for expert e lands at grouped row
// seg_off[r][j][s] + (i - expert_send_off[s][e]) of rank r = e / Er.
struct GroupedDest {
    int N, E, cap;
    const int32_t *idx, *eso, *seg_off;
    uint8_t *grp_q;
    float *grp_s;
    int32_t *grp_src;
};

// Send row and grouped row of assignment k of token tok (-1: none).
template <bool kGrouped>
__device__ __forceinline__ void dest_rows(long long tok, int k, int T, int R, long long TR,
                                          const int32_t *__restrict__ slot_row,
                                          const GroupedDest &gd, long long &row,
                                          long long &grow) {
    const long long s = div_nonneg(tok, T);
    const int sr = __ldg(slot_row + tok * R + k);
    row = (sr >= 0 && sr < TR) ? s * TR + sr : -1;
    grow = -1;
    if (kGrouped && row >= 0) {
        const int e = __ldg(gd.idx + tok * R + k);
        if ((unsigned)e < (unsigned)gd.E) {
            const int Er = gd.E / gd.N, r = e / Er, j = e - r * Er;
            const int g = __ldg(gd.seg_off + ((size_t)r * Er + j) * gd.N + s) +
                          (sr - __ldg(gd.eso + (size_t)s * (gd.E + 1) + e));
            if (g >= 0 && g < gd.cap) grow = (long long)r * gd.cap + g;
        }
    }
}

// Publication of the send rows by (sender s, receiver r) group, for the
// signalled dispatch: each (row, piece) written adds one to cnt[s][r] after
// a release fence; the writer that brings the count to the group's size
// (rows of s for r, times the pieces per row) fences once more and sets
// published[s][r] = 1.
struct Signal {
    int N, Er, npieces;
    const int32_t *idx;       // [N][T][R] expert ids
    const int32_t *send_off;  // [N][N+1] per-peer send offsets
    int32_t *cnt;             // [N][N] (row, piece) pairs written
    int32_t *published;       // [N][N] 1 once the group is complete
};

// Thread k of the CTA publishes its row of an item whose stores are issued.
__device__ __forceinline__ void publish_row(const Signal &sg, int g, int target) {
    __threadfence();
    if (atomicAdd(sg.cnt + g, 1) + 1 == target) {
        __threadfence();
        st_release(sg.published + g, 1);
    }
}

// kHostX: x is pinned host memory, read by the threads with 16-byte loads
// over the CPU-GPU link (zero copy) instead of by bulk copies.
// kDest == kLowLatency: send_q / send_s / send_tok are the low-latency rows,
// scales and source ids, and each item's rows are found by the CTA itself
// (no routing kernel before it).
// kSignal: publish every row written (Signal above) once the item's stores
// are issued: the barrier that ends the item orders every thread's stores
// before the publishing thread's release fence.
// The CTA handles items cta, cta + ncta, ...
// Returns the number of items the CTA processed, or -1 after a timeout.
template <Dest kDest, bool kHostX, bool kSignal = false, class Gate = NoGate>
__device__ __forceinline__ int quant_pack_body(
    int T, int R, int H, int P, long long tok0, long long nitems, const uint16_t *__restrict__ x,
    const int32_t *__restrict__ slot_row, uint8_t *__restrict__ send_q, float *__restrict__ send_s,
    int32_t *__restrict__ send_tok, int32_t *__restrict__ status, const GroupedDest &gd,
    const LLDest &ll, const Signal &sg, long long cta, long long ncta, const Gate &gate = Gate()) {
    constexpr bool kGrouped = kDest == Dest::kSendGrouped;
    constexpr bool kLL = kDest == Dest::kLowLatency;
    constexpr bool kLLR = kDest == Dest::kLowLatencyRanked;
    constexpr int kXStages = x_stages(kDest, kSignal);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *sm = align128(smem_raw);
    uint16_t *xbuf = reinterpret_cast<uint16_t *>(sm);  // [2][P] bf16
    __shared__ uint64_t xbar[kXStages];
    __shared__ long long rows[MOE_MAX_TOPK];   // destination rows of the current item
    __shared__ long long grows[MOE_MAX_TOPK];  // and its grouped rows (kGrouped)
    __shared__ int wpart[8][MOE_MAX_TOPK];  // LL: per-warp counts of earlier equal ids
    int *hist = reinterpret_cast<int *>(sm + stage_bytes(P, kXStages));  // [E], LL

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
    const int Sb = H >> 7, npieces = (H + P - 1) / P;
    const long long TR = (long long)T * R;

    if (tid == 0) {
        for (int b = 0; b < kXStages; ++b) mbar_init(&xbar[b], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // host x: the threads copy the piece with 16-byte loads
    auto host_copy = [&](long long item, int b) {
        const long long tok = tok0 + div_nonneg(item, npieces);
        const int off = (int)(item - div_nonneg(item, npieces) * npieces) * P;
        const int len = min(P, H - off);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + tok * H + off);
        uint4 *dst = reinterpret_cast<uint4 *>(xbuf + (size_t)b * P);
        for (int i = threadIdx.x; i < (len >> 3); i += blockDim.x) dst[i] = src[i];
    };
    auto issue_load = [&](long long item, int b) {
        const long long tok = tok0 + div_nonneg(item, npieces);
        const int off = (int)(item - div_nonneg(item, npieces) * npieces) * P;
        const int len = min(P, H - off);
        mbar_arrive_expect_tx(&xbar[b], (uint32_t)len * 2u);
        bulk_g2s(xbuf + (size_t)b * P, x + tok * H + off, (uint32_t)len * 2u, &xbar[b]);
    };

    const long long first = cta, G = ncta;
    // the first kXStages - 1 pieces; with a gate every buffer's piece before
    // it, past which everything that another kernel or phase writes is read
    constexpr int kPre = Gate::kPrefetch ? kXStages : kXStages - 1;
    if (!kHostX && tid == 0)
        for (int i = 0; i < kPre && first + (long long)i * G < nitems; ++i)
            issue_load(first + (long long)i * G, i);
    if constexpr (kHostX && Gate::kPrefetch) {
        // host x is no output of the kernel before the gate either: every
        // buffer's piece crosses the link while that kernel runs
        for (int i = 0; i < kXStages && first + (long long)i * G < nitems; ++i)
            host_copy(first + (long long)i * G, i);
        __syncthreads();
    }
    if constexpr (Gate::kPrefetch) gate(reinterpret_cast<int *>(sm + stage_bytes(P, kXStages)));
    bool timed_out = false;
    // thread tid < R: destinations of the current item, read one item ahead
    long long prow = -1, pgrow = -1;
    auto next_rows = [&](long long item) {
        const long long tok = tok0 + div_nonneg(item, npieces);
        if constexpr (kLLR) {
            // the low-latency row ranked by this kernel (read through L2)
            prow = __ldcg(ll.ll_row + tok * R + tid);
        } else {
            dest_rows<kGrouped>(tok, tid, T, R, TR, slot_row, gd, prow, pgrow);
        }
    };
    if (!kLL && tid < R && first < nitems) next_rows(first);

    int n = 0, b = 0;   // item count, its buffer (n mod kXStages)
    uint32_t par = 0;   // phase parity of buffer b's barrier: (n / kXStages) & 1
    for (long long item = first; item < nitems;
         item += G, ++n, b = (b + 1 == kXStages) ? 0 : b + 1, par ^= (b == 0) ? 1u : 0u) {
        const long long tok = tok0 + div_nonneg(item, npieces);
        const int piece = (int)(item - (tok - tok0) * npieces);
        const int off = piece * P, len = min(P, H - off), nch = len >> 4;
        const long long s = div_nonneg(tok, T);
        const int t = (int)(tok - s * T);
        // the piece kXStages - 1 items ahead, into the buffer the previous
        // item released (already issued before the gate when n == 0)
        const long long ahead = item + (long long)(kXStages - 1) * G;
        if (!kHostX && tid == 0 && ahead < nitems && !(Gate::kPrefetch && n == 0))
            issue_load(ahead, b == 0 ? kXStages - 1 : b - 1);
        if constexpr (kLL) {
            // rows of this token in the low-latency layout, while x arrives:
            // u_k = earlier assignments of rank s with the same expert, eight
            // slots at a time, counted in registers and summed per warp
            const int32_t *ids = ll.idx + s * TR;
            const int lim = t * R + R - 1;  // flat indices before the last slot
            for (int k0 = 0; k0 < R; k0 += 8) {
                int ekr[8], c[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    ekr[u] = k0 + u < R ? __ldg(ll.idx + tok * R + k0 + u) : 0;
                    c[u] = 0;
                }
                for (int i = tid; i < lim; i += nthr) {
                    const int v = __ldg(ids + i);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        c[u] += (k0 + u < R && v == ekr[u] && i < t * R + k0 + u) ? 1 : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int tot = (int)__reduce_add_sync(kFull, (unsigned)c[u]);
                    if (lane == 0 && k0 + u < R) wpart[warp][k0 + u] = tot;
                }
            }
            if (t == 0 && piece == 0) {  // region counts of rank s, once
                for (int e = tid; e < ll.E; e += nthr) hist[e] = 0;
                __syncthreads();
                int bad = 0;
                for (int i = tid; i < TR; i += nthr) {
                    const int v = __ldg(ids + i);
                    if ((unsigned)v < (unsigned)ll.E)
                        atomicAdd(&hist[v], 1);
                    else
                        bad = 1;
                }
                if (__syncthreads_or(bad) && tid == 0) flag(status, MOE_ST_BAD_EXPERT);
                int over = 0;
                for (int e = tid; e < ll.E; e += nthr) {
                    ll.ll_count[(size_t)e * ll.N + s] = hist[e];  // region (e / Er, e % Er, s)
                    over |= hist[e] > T;
                }
                if (__syncthreads_or(over) && tid == 0) flag(status, MOE_ST_CAPACITY);
            }
            __syncthreads();
            if (tid < R) {
                const int e = __ldg(ll.idx + tok * R + tid);
                int u = 0;
                for (int w = 0; w < (nthr >> 5); ++w) u += wpart[w][tid];
                const long long row =
                    ((unsigned)e < (unsigned)ll.E && u < T) ? ((long long)e * ll.N + s) * T + u : -1;
                prow = row;
                if (piece == 0) ll.ll_row[tok * R + tid] = (int32_t)row;
            }
        }
        // the rows every thread stores to, visible after the barrier below
        if (tid < R) {
            rows[tid] = prow;
            grows[tid] = pgrow;
        }
        if constexpr (kHostX) {
            if (!(Gate::kPrefetch && n < kXStages)) host_copy(item, b);
            __syncthreads();
        } else {
            const bool ok = mbar_wait(&xbar[b], par);
            if (__syncthreads_or(!ok)) {
                timed_out = true;
                break;
            }
        }

        const uint16_t *xs = xbuf + (size_t)b * P;
        for (int cb = warp * 32; cb < nch; cb += nthr) {
            const int c = cb + lane;
            const bool in = c < nch;
            uint4 va = make_uint4(0, 0, 0, 0), vb = va;
            if (in) {
                const uint4 *p = reinterpret_cast<const uint4 *>(xs + (size_t)c * 16);
                va = p[0];
                vb = p[1];
            }
            float amax = amax16(va, vb);
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
            const float scale = __fdiv_rn(amax, 448.0f);
            const uint4 q = amax > 0.0f ? quant16(va, vb, scale) : make_uint4(0, 0, 0, 0);
            if (in) {
                const int sc = (off >> 7) + (c >> 3);
                for (int k = 0; k < R; ++k) {
                    const long long row = rows[k];
                    if (row >= 0) {
                        uint4 *d = reinterpret_cast<uint4 *>(send_q + row * H + off + c * 16);
                        if constexpr (kDest == Dest::kSend)
                            *d = q;  // read back soon after (receive pull, signalled copy)
                        else
                            __stcs(d, q);
                        if ((c & 7) == 0) send_s[row * Sb + sc] = scale;
                    }
                    if constexpr (kGrouped) {
                        const long long grow = grows[k];
                        if (grow >= 0) {
                            __stcs(reinterpret_cast<uint4 *>(gd.grp_q + grow * H + off + c * 16), q);
                            if ((c & 7) == 0) gd.grp_s[grow * Sb + sc] = scale;
                        }
                    }
                }
            }
        }
        // every store of this item is issued and buffer b is read
        __syncthreads();
        if (tid < R) {
            const long long row = rows[tid];
            if (piece == 0 && row >= 0) {
                send_tok[row] = t;
                if (kGrouped && grows[tid] >= 0)
                    *reinterpret_cast<int2 *>(gd.grp_src + grows[tid] * 2) = make_int2((int)s, t);
            }
            if constexpr (kSignal) {
                const int e = row >= 0 ? __ldg(sg.idx + tok * R + tid) : -1;
                if ((unsigned)e < (unsigned)(sg.N * sg.Er)) {
                    const int r = e / sg.Er;
                    const int32_t *so = sg.send_off + s * (sg.N + 1);
                    publish_row(sg, (int)s * sg.N + r,
                                (__ldg(so + r + 1) - __ldg(so + r)) * sg.npieces);
                }
            }
            // the next item's destinations
            if (!kLL && item + G < nitems) next_rows(item + G);
        }
    }
    if (tid == 0 && timed_out) {
        flag(status, MOE_ST_TIMEOUT);
        // let every issued load (items n .. n + kXStages - 1) land before
        // shared memory goes away
        for (int i = n; i < n + kXStages; ++i)
            if (first + (long long)i * G < nitems)
                mbar_wait(&xbar[i % kXStages], (uint32_t)((i / kXStages) & 1));
    }
    return timed_out ? -1 : n;
}

// kPdl: launched as the programmatic dependent of the routing kernel (the
// fused dispatch of moe_dispatch): both x buffers are filled before
// griddepcontrol.wait, so the first pieces arrive while the routing kernel
// runs; nothing the routing kernel writes is read, and nothing is written,
// before the wait.
// At most MOE_QUANT_MAXNREG registers per thread, so that five 224-thread
// CTAs (a 7168-element row in 3584-element pieces, 16 elements a thread,
// or whole rows in two passes) fit on an SM.
#ifndef MOE_QUANT_MAXNREG
#define MOE_QUANT_MAXNREG 56
#endif
template <Dest kDest, bool kHostX, bool kPdl = false>
__global__ void __maxnreg__(MOE_QUANT_MAXNREG)
    k_quant_pack_staged(int T, int R, int H, int P, long long tok0, long long nitems,
                        const uint16_t *__restrict__ x, const int32_t *__restrict__ slot_row,
                        uint8_t *__restrict__ send_q, float *__restrict__ send_s,
                        int32_t *__restrict__ send_tok, int32_t *__restrict__ status,
                        const GroupedDest gd, const LLDest ll) {
    const Signal sg = {};
    if constexpr (kPdl)
        quant_pack_body<kDest, kHostX, false, PdlGate>(T, R, H, P, tok0, nitems, x, slot_row,
                                                       send_q, send_s, send_tok, status, gd, ll,
                                                       sg, blockIdx.x, gridDim.x);
    else
        quant_pack_body<kDest, kHostX>(T, R, H, P, tok0, nitems, x, slot_row, send_q, send_s,
                                       send_tok, status, gd, ll, sg, blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------ ranked low-latency dispatch
//
// The low-latency dispatch for longer batches, in one co-resident grid.
// First every sender's ids are ranked once: CTA c takes senders c, c + G,
// ... and runs the routing kernels' counting pass over them (per-warp tables
// in shared memory, see sender_count); the row of assignment (t, k) of
// sender s with expert e is region (e, s), row u = the number of earlier
// assignments of s to e, or none when u >= T (MOE_ST_CAPACITY); ll_count
// gets every region's count.  The x loads of each CTA's first two items are
// already in flight.  Then the grid meets at a grid-wide barrier and
// quantises and packs as the staged kernel does, each item's rows read from
// ll_row.  This replaces the per-token search of earlier ids (work T*R per
// token) by one pass over each sender's ids.
struct LLRankGate {
    static constexpr bool kPrefetch = true;
    int N, T, E, R;
    LLDest ll;
    int32_t *status;
    __device__ __forceinline__ void operator()(int *tables) const {
        const int tid = threadIdx.x, TR = T * R;
        for (int s = blockIdx.x; s < N; s += gridDim.x) {
            int rk[kAhead];
            SenderShare sh;
            // pass-1 ranks of long shares are kept in ll_row[s] until rewritten below
            const bool bad = sender_count(N, T, E, R, s, ll.idx, ll.ll_row, tables, rk, sh);
            int over = 0;
            for (int e = tid; e < E; e += blockDim.x) {
                const int c = tables[e + 1] - tables[e];
                ll.ll_count[(size_t)e * N + s] = c;  // region (e / Er, e % Er, s)
                over |= c > T;
            }
            int32_t *row = ll.ll_row + (size_t)s * TR;
            sender_ranks(T, E, R, s, ll.idx, ll.ll_row, tables, rk, sh, [&](int i, int e, int u) {
                row[i] = (e >= 0 && u < T) ? (int32_t)(((long long)e * N + s) * T + u) : -1;
            });
            if (__syncthreads_or(over) && tid == 0) flag(status, MOE_ST_CAPACITY);
            if (bad && tid == 0) flag(status, MOE_ST_BAD_EXPERT);
        }
        cooperative_groups::this_grid().sync();
    }
};

#ifndef MOE_LL_RANKED_MINB
#define MOE_LL_RANKED_MINB 4
#endif
template <bool kHostX>
__global__ void __launch_bounds__(256, MOE_LL_RANKED_MINB)
    k_dispatch_ll_ranked(int T, int R, int H, int P, long long nitems,
                         const uint16_t *__restrict__ x, uint8_t *__restrict__ ll_q,
                         float *__restrict__ ll_s, int32_t *__restrict__ ll_src,
                         int32_t *__restrict__ status, const LLDest ll, int E) {
    const GroupedDest gd = {};
    const Signal sg = {};
    LLRankGate gate;
    gate.N = ll.N;
    gate.T = T;
    gate.E = E;
    gate.R = R;
    gate.ll = ll;
    gate.status = status;
    quant_pack_body<Dest::kLowLatencyRanked, kHostX, false, LLRankGate>(
        T, R, H, P, 0, nitems, x, nullptr, ll_q, ll_s, ll_src, status, gd, ll, sg, blockIdx.x,
        gridDim.x, gate);
}

// ------------------------------------------------------------ signalled dispatch
//
// Dispatch send and receive shuffle in one co-resident grid, handing rows
// over by per-group arrival flags instead of a kernel boundary (the
// decoupled signalling of "MoE multi-node inference bottleneck overturned:
// Perseus removes hidden serialization", section 3, Algorithm 1 and
// Figure 6: transfers first, then one fence and one signal per destination
// group, issued by whichever participant completes the group).
// Every CTA first quantises + packs its (token, piece) items into the send
// buffers (items in order, so senders complete roughly in order), publishing
// each (sender, receiver) group as its rows complete; then it pulls its
// contiguous range of send rows into the grouped layout, each row waiting
// (bounded) until its group is published -- a CTA that finishes packing
// early starts on the groups already complete while others still pack.
// The last CTA to finish clears the counters and flags, so the scratch is
// zero again for the next call.  Registers are capped at 64 (four CTAs per
// SM; the pull moves 4 vectors per lane per step to stay within the cap):
// five or six CTAs per SM, or 3 CTAs with 8 vectors, measured the same or
// slower.
#ifndef MOE_SIG_VECS
#define MOE_SIG_VECS 4
#endif
#ifndef MOE_SIG_MINB
#define MOE_SIG_MINB 4
#endif

template <bool kHostX>
__global__ void __launch_bounds__(256, MOE_SIG_MINB)
    k_dispatch_signalled(int T, int R, int H, int P, long long nitems,
                         const uint16_t *__restrict__ x, const int32_t *__restrict__ slot_row,
                         uint8_t *__restrict__ send_q, float *__restrict__ send_s,
                         int32_t *__restrict__ send_tok, int32_t *__restrict__ status,
                         const DispatchMapT<true> pull, const Signal sg, int32_t *done) {
    {
        const GroupedDest gd = {};
        const LLDest ll = {};
        quant_pack_body<Dest::kSend, kHostX, true>(T, R, H, P, 0, nitems, x, slot_row, send_q,
                                                   send_s, send_tok, status, gd, ll, sg,
                                                   blockIdx.x, gridDim.x);
    }
    {
        const long long nrows = (long long)pull.N * pull.TR;
        const int nw = blockDim.x >> 5;
        const long long W = (long long)gridDim.x * nw;
        const long long gw = (long long)blockIdx.x * nw + (threadIdx.x >> 5);
        const long long per = (nrows + W - 1) / W;
        const long long r0 = gw * per, r1 = min(nrows, r0 + per);
        if (r0 < r1) copy_rows<MOE_SIG_VECS>(pull, 0, r0, r1);
    }
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (last) {
        __threadfence();
        const int n2 = sg.N * sg.N;
        for (int i = threadIdx.x; i < n2; i += blockDim.x) {
            sg.cnt[i] = 0;
            sg.published[i] = 0;
        }
        if (threadIdx.x == 0) *done = 0;
    }
}

static int quant_threads(int nch) {
    // a block size that divides the piece's 16-element chunks into whole passes
    for (int w = 8; w >= 1; --w)
        if (nch % (32 * w) == 0) return 32 * w;
    return nch >= 256 ? 256 : 32 * ((nch + 31) / 32);
}

// Pinned host memory (reachable from the GPU through unified addressing)?
static bool is_host_memory(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// Piece length: rows split into the fewest pieces of at most `cap`
// elements, of equal length (multiples of 128); a batch with fewer pieces
// than four per SM gets shorter ones (at least MOE_MIN_PIECE elements), so
// that its few tokens spread over more CTAs.
#ifndef MOE_MIN_PIECE
#define MOE_MIN_PIECE 1024
#endif
static_assert(MOE_MIN_PIECE % 128 == 0, "pieces hold whole scale blocks");
static int piece_elems(long long ntok, int H, int cap) {
    const int np = (H + cap - 1) / cap;
    const int P = ((H + np - 1) / np + 127) / 128 * 128;
    const long long want = (long long)sm_count() * 4;
    if (ntok <= 0 || ntok * ((H + P - 1) / P) >= want) return P;
    const long long per_tok = (want + ntok - 1) / ntok;
    long long q = (H + per_tok - 1) / per_tok;
    q = (q + 127) / 128 * 128;
    if (q < MOE_MIN_PIECE) q = MOE_MIN_PIECE;
    return q < P ? (int)q : P;
}

template <Dest kDest, bool kHostX, bool kPdl>
static cudaError_t launch_staged_x(const moe_shape &sh, const uint16_t *x,
                                   const int32_t *slot_row, uint8_t *send_q, float *send_s,
                                   int32_t *send_tok, int32_t *status, const GroupedDest &gd,
                                   const LLDest &ll, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    auto kern = k_quant_pack_staged<kDest, kHostX, kPdl>;
    constexpr int kNB = x_stages(kDest, false);
    // a long batch: more than MOE_PACK_LONG tokens per CTA of five per SM
    const bool long_batch = ntok > (long long)MOE_PACK_LONG * 5 * sm_count();
    const int cap = piece_cap(kDest, false, long_batch);
    const int P = piece_elems(ntok, sh.H, cap);
    const long long nitems = ntok * ((sh.H + P - 1) / P);
    const int threads = quant_threads(P / 16);
    constexpr int kHist = kDest == Dest::kLowLatency ? MOE_MAX_EXPERTS * 4 : 0;
    const int smem = (int)stage_bytes(P, kNB) + 128 + kHist;
    static LaunchMemo memo;
    int occ = 1;
    cudaError_t err = memo.get(((long long)smem << 16) | threads, &occ, [&](int *v) {
        // the attribute allows the largest piece, whatever this call's P
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)stage_bytes(kPieceElems, kNB) + 128 + kHist);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, smem);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    long long grid = (long long)sm_count() * occ;
    if (grid > nitems) grid = nitems;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = kPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, sh.T, sh.R, sh.H, P, 0LL, nitems, x, slot_row, send_q,
                              send_s, send_tok, status, gd, ll);
}

template <Dest kDest, bool kPdl = false>
static cudaError_t launch_staged(const moe_shape &sh, const uint16_t *x, const int32_t *slot_row,
                                 uint8_t *send_q, float *send_s, int32_t *send_tok,
                                 int32_t *status, const GroupedDest &gd, const LLDest &ll,
                                 cudaStream_t st) {
    if ((long long)sh.N * sh.T <= 0) return cudaSuccess;
    if (is_host_memory(x))
        return launch_staged_x<kDest, true, kPdl>(sh, x, slot_row, send_q, send_s, send_tok,
                                                  status, gd, ll, st);
    return launch_staged_x<kDest, false, kPdl>(sh, x, slot_row, send_q, send_s, send_tok, status,
                                               gd, ll, st);
}

cudaError_t launch_quant_pack(const moe_shape &sh, const uint16_t *x, const int32_t *slot_row,
                              uint8_t *send_q, float *send_s, int32_t *send_tok, int32_t *status,
                              cudaStream_t st) {
    GroupedDest gd = {};
    LLDest ll = {};
    return launch_staged<Dest::kSend>(sh, x, slot_row, send_q, send_s, send_tok, status, gd, ll,
                                      st);
}

// The ranked low-latency dispatch: one co-resident grid (the grid-wide
// barrier between ranking and packing needs every CTA resident).
template <bool kHostX>
static cudaError_t launch_ll_ranked_x(const moe_shape &sh, const uint16_t *x, uint8_t *ll_q,
                                      float *ll_s, int32_t *ll_src, int32_t *status,
                                      const LLDest &ll, cudaStream_t st) {
    const long long ntok = (long long)sh.N * sh.T;
    auto kern = k_dispatch_ll_ranked<kHostX>;
    constexpr int kNB = x_stages(Dest::kLowLatencyRanked, false);
    const int P = piece_elems(ntok, sh.H, piece_cap(Dest::kLowLatencyRanked, false));
    const long long nitems = ntok * ((sh.H + P - 1) / P);
    const int threads = quant_threads(P / 16);
    // x buffers, then the counting tables of one sender: [E+1] + [warps][E] ints
    const auto tables = [](int E, int thr) { return (size_t)(E + 1 + (thr / 32) * E) * 4; };
    const int smem = (int)(stage_bytes(P, kNB) + 128 + tables(sh.E, threads));
    static LaunchMemo memo;
    int occ = 0;
    cudaError_t err = memo.get(((long long)smem << 16) | threads, &occ, [&](int *v) {
        cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)(stage_bytes(kPieceElems, kNB) + 128 + tables(MOE_MAX_EXPERTS, 256)));
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, smem);
        return e;
    });
    if (err != cudaSuccess) return err;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)sm_count() * occ;
    if (grid > nitems) grid = nitems;
    return launch_kernel_coresident(kern, dim3((unsigned)grid), dim3(threads), (size_t)smem, st,
                                    sh.T, sh.R, sh.H, P, nitems, x, ll_q, ll_s, ll_src, status, ll,
                                    sh.E);
}

// Batches of more than MOE_LL_SEARCH_MAX ids per rank rank every sender's ids
// once (k_dispatch_ll_ranked); shorter ones let each CTA count its token's
// earlier ids itself, which needs no grid-wide barrier.  Measured: at 1024
// ids per rank (DSv3 EP16, Kimi-K2 EP32) the per-token count took 34.3 and
// 58.6 us against 42.5 and 70.9 ranked; at 4096 (Qwen3-30B EP16, 512
// tokens) 68.1 against 59.8 ranked.
#ifndef MOE_LL_SEARCH_MAX
#define MOE_LL_SEARCH_MAX 2048
#endif

cudaError_t launch_dispatch_ll(const moe_shape &sh, const uint16_t *x, const int32_t *idx,
                               uint8_t *ll_q, float *ll_s, int32_t *ll_src, int32_t *ll_count,
                               int32_t *ll_row, int32_t *status, cudaStream_t st) {
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return err;
    GroupedDest gd = {};
    LLDest ll;
    ll.N = sh.N;
    ll.E = sh.E;
    ll.idx = idx;
    ll.ll_row = ll_row;
    ll.ll_count = ll_count;
    // an empty batch: every region is empty (the kernels write the counts
    // from each sender's token 0, and there is none)
    if ((long long)sh.N * sh.T <= 0)
        return cudaMemsetAsync(ll_count, 0, (size_t)sh.N * sh.E * sizeof(int32_t), st);
    if ((long long)sh.T * sh.R > MOE_LL_SEARCH_MAX) {
        if (is_host_memory(x))
            return launch_ll_ranked_x<true>(sh, x, ll_q, ll_s, ll_src, status, ll, st);
        return launch_ll_ranked_x<false>(sh, x, ll_q, ll_s, ll_src, status, ll, st);
    }
    return launch_staged<Dest::kLowLatency>(sh, x, nullptr, ll_q, ll_s, ll_src, status, gd, ll,
                                            st);
}

template <bool kHostX>
static cudaError_t launch_signalled_x(const moe_shape &sh, int cap, const uint16_t *x,
                                      const int32_t *idx, const int32_t *slot_row,
                                      const int32_t *send_off, const int32_t *eso,
                                      const int32_t *seg_off, uint8_t *send_q, float *send_s,
                                      int32_t *send_tok, uint8_t *grp_q, float *grp_s,
                                      int32_t *grp_src, int32_t *sig, int32_t *status,
                                      cudaStream_t st) {
    auto kern = k_dispatch_signalled<kHostX>;
    constexpr int kNB = x_stages(Dest::kSend, true);
    const int P = piece_elems((long long)sh.N * sh.T, sh.H, piece_cap(Dest::kSend, true));
    const int npieces = (sh.H + P - 1) / P;
    const long long nitems = (long long)sh.N * sh.T * npieces;
    const int threads = quant_threads(P / 16);
    const int smem = (int)stage_bytes(P, kNB) + 128;
    static LaunchMemo memo;
    int occ = 1;
    cudaError_t err = memo.get(((long long)smem << 16) | threads, &occ, [&](int *v) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)stage_bytes(kPieceElems, kNB) + 128);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, kern, threads, smem);
        if (*v < 1) *v = 1;
        return e;
    });
    if (err != cudaSuccess) return err;
    // every CTA resident at once: rows wait on groups other CTAs pack
    long long grid = (long long)sm_count() * occ;
    if (grid > nitems) grid = nitems;
    const int N = sh.N;
    Signal sg;
    sg.N = N;
    sg.Er = sh.E / N;
    sg.npieces = npieces;
    sg.idx = idx;
    sg.send_off = send_off;
    sg.cnt = sig;
    sg.published = sig + (size_t)N * N;
    DispatchMapT<true> m;
    m.N = N;
    m.E = sh.E;
    m.Er = sh.E / N;
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
    m.published = sg.published;
    m.status = status;
    return launch_kernel_coresident(kern, dim3((unsigned)grid), dim3(threads), (size_t)smem, st,
                                    sh.T, sh.R, sh.H, P, nitems, x, slot_row, send_q,
                                    send_s, send_tok, status, m, sg, sig + 2 * (size_t)N * N);
}

cudaError_t launch_dispatch_signalled(const moe_shape &sh, int cap, const uint16_t *x,
                                      const int32_t *idx, const int32_t *slot_row,
                                      const int32_t *send_off, const int32_t *eso,
                                      const int32_t *seg_off, uint8_t *send_q, float *send_s,
                                      int32_t *send_tok, uint8_t *grp_q, float *grp_s,
                                      int32_t *grp_src, int32_t *sig, int32_t *status,
                                      cudaStream_t st) {
    if ((long long)sh.N * sh.T <= 0) return cudaSuccess;
    if (is_host_memory(x))
        return launch_signalled_x<true>(sh, cap, x, idx, slot_row, send_off, eso, seg_off, send_q,
                                        send_s, send_tok, grp_q, grp_s, grp_src, sig, status, st);
    return launch_signalled_x<false>(sh, cap, x, idx, slot_row, send_off, eso, seg_off, send_q,
                                     send_s, send_tok, grp_q, grp_s, grp_src, sig, status, st);
}

// moe_dispatch launches the fused dispatch as the programmatic dependent of
// its routing kernel (after_route): the first pieces of x load while the
// routing kernel runs.  On the DSv3 EP16 layer (CUDA graph) this measured
// X us against Y us.
#ifndef MOE_DISPATCH_PDL
#define MOE_DISPATCH_PDL 1
#endif

cudaError_t launch_dispatch_fused(const moe_shape &sh, int cap, const uint16_t *x,
                                  const int32_t *idx, const int32_t *slot_row, const int32_t *eso,
                                  const int32_t *seg_off, uint8_t *send_q, float *send_s,
                                  int32_t *send_tok, uint8_t *grp_q, float *grp_s,
                                  int32_t *grp_src, int32_t *status, cudaStream_t st,
                                  bool after_route) {
    GroupedDest gd;
    gd.N = sh.N;
    gd.E = sh.E;
    gd.cap = cap;
    gd.idx = idx;
    gd.eso = eso;
    gd.seg_off = seg_off;
    gd.grp_q = grp_q;
    gd.grp_s = grp_s;
    gd.grp_src = grp_src;
    LLDest ll = {};
    if (after_route && MOE_DISPATCH_PDL)
        return launch_staged<Dest::kSendGrouped, true>(sh, x, slot_row, send_q, send_s, send_tok,
                                                       status, gd, ll, st);
    return launch_staged<Dest::kSendGrouped>(sh, x, slot_row, send_q, send_s, send_tok, status, gd,
                                             ll, st);
}

}  // namespace moe
