// pipeline.cu -- moe_dispatch / moe_combine: the whole dispatch and combine
// as one call each, ordered by chunks of sender ranks so that each consumer
// kernel reads its producer's rows from L2.
//
// A chunk is a run of consecutive ranks [s0, s1).  Dispatch: quantise and
// pack the tokens of those ranks (send rows [s0*T*R, s1*T*R)), then pull
// exactly those send rows into the grouped layout.  Combine: pack the output
// rows that go back to those ranks (the same flat send-row range, seen from
// the expert side), then reduce their tokens.
//
// Measured on GB300 inside a CUDA graph, neither chunking nor programmatic
// dependent launch (starting a kernel during its predecessor's tail) beat the
// plain sequence, so the default is one chunk and normal launches.
#include <cstdint>

#include "launch.h"
#include "moeroute.h"

namespace {

// chunks >= 1: that many (at most N); chunks == 0: one chunk.  Measured on
// GB300, every extra kernel launch costs more than the L2 re-reads it saves
// (each launch pays its ramp-up and tail), so the default does not split.
int chunk_count(int N, long long bytes_per_rank, int chunks) {
    (void)bytes_per_rank;
    if (chunks >= 1) return chunks < N ? chunks : N;
    return 1;
}

bool aligned(const void *p, long long bytes) {
    return bytes == 0 || (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0);
}

}  // namespace

extern "C" int moe_dispatch(const moe_shape *sh, const moe_buffers *b, int chunks, void *stream) {
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!b || chunks < 0) return MOE_EINVAL;
    if (!aligned(b->topk_idx, z.bytes_topk_idx) || !aligned(b->x, z.bytes_x) ||
        !aligned(b->expert_count, z.bytes_expert_count) || !aligned(b->send_off, z.bytes_send_off) ||
        !aligned(b->expert_send_off, z.bytes_expert_send_off) ||
        !aligned(b->slot_row, z.bytes_topk_idx) || !aligned(b->grp_off, z.bytes_grp_off) ||
        !aligned(b->seg_off, z.bytes_seg_off) || !aligned(b->csend_off, z.bytes_send_off) ||
        !aligned(b->m_sizes, z.bytes_m_sizes) || !aligned(b->send_q, z.bytes_send_q) ||
        !aligned(b->send_s, z.bytes_send_s) || !aligned(b->send_tok, z.bytes_send_tok) ||
        !aligned(b->grp_q, z.bytes_grp_q) || !aligned(b->grp_s, z.bytes_grp_s) ||
        !aligned(b->grp_src, z.bytes_grp_src) || !aligned(b->status, 4))
        return MOE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int cap = (int)z.cap;
    if (moe::launch_route(*sh, cap, b->topk_idx, b->expert_count, b->send_off, b->expert_send_off,
                          b->slot_row, b->grp_off, b->seg_off, b->csend_off, b->m_sizes, b->status,
                          st) != cudaSuccess)
        return MOE_ECUDA;
    const long long TR = (long long)sh->T * sh->R;
    const int C = chunk_count(sh->N, TR * (sh->H + sh->H / 32), chunks);
    for (int c = 0; c < C; ++c) {
        const long long s0 = (long long)sh->N * c / C, s1 = (long long)sh->N * (c + 1) / C;
        if (s0 == s1) continue;
        if (moe::launch_quant_pack(*sh, b->x, b->slot_row, b->send_q, b->send_s, b->send_tok,
                                   b->status, st, s0 * sh->T, s1 * sh->T) != cudaSuccess)
            return MOE_ECUDA;
        if (moe::launch_dispatch_pull(*sh, cap, b->send_q, b->send_s, b->send_tok,
                                      b->expert_send_off, b->seg_off, b->grp_q, b->grp_s,
                                      b->grp_src, b->status, st, s0 * TR, s1 * TR) != cudaSuccess)
            return MOE_ECUDA;
    }
    return MOE_OK;
}

extern "C" int moe_combine(const moe_shape *sh, const moe_buffers *b, int chunks, void *stream) {
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!b || chunks < 0) return MOE_EINVAL;
    if (!aligned(b->topk_idx, z.bytes_topk_idx) || !aligned(b->topk_w, z.bytes_topk_idx) ||
        !aligned(b->y, z.bytes_y) || !aligned(b->expert_send_off, z.bytes_expert_send_off) ||
        !aligned(b->send_off, z.bytes_send_off) || !aligned(b->slot_row, z.bytes_topk_idx) ||
        !aligned(b->seg_off, z.bytes_seg_off) || !aligned(b->csend_off, z.bytes_send_off) ||
        !aligned(b->csend, z.bytes_y) || !aligned(b->out, z.bytes_x) || !aligned(b->status, 4))
        return MOE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int cap = (int)z.cap;
    const long long TR = (long long)sh->T * sh->R;
    const int C = chunk_count(sh->N, TR * 2LL * sh->H, chunks);
    for (int c = 0; c < C; ++c) {
        const long long s0 = (long long)sh->N * c / C, s1 = (long long)sh->N * (c + 1) / C;
        if (s0 == s1) continue;
        if (moe::launch_combine_pack(*sh, cap, b->y, b->expert_send_off, b->send_off, b->seg_off,
                                     b->csend_off, b->csend, b->status, st, s0 * TR, s1 * TR) != cudaSuccess)
            return MOE_ECUDA;
        if (moe::launch_combine_reduce(*sh, cap, b->csend, b->topk_idx, b->topk_w, b->slot_row,
                                       b->send_off, b->csend_off, b->out, st, s0 * sh->T,
                                       s1 * sh->T) != cudaSuccess)
            return MOE_ECUDA;
    }
    return MOE_OK;
}
