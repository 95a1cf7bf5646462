// pipeline.cu -- moe_dispatch / moe_combine: the whole dispatch and the
// whole combine as one call each, built from the fused kernels.
//
// moe_dispatch: k_route (route_count + exchange), then one pass that
//   quantises each token once and writes its fp8 rows both to the send
//   buffer and to their grouped rows.  Every output of the separate calls is
//   produced; the receive shuffle's re-read of the send buffer is not needed
//   because the grouped rows are written from the same shared-memory copy.
// moe_combine: one pass that reads each expert-output row once from y,
//   writes it to its combine send row and accumulates it into the token's
//   output.  The combine send buffer is produced exactly as by
//   moe_combine_send; reading it back is not needed.
//
// On the pages the sender learns every receiver's offsets from the routing
// exchange and then writes its tokens straight to their places ("Send and
// receive buffers"); with all ranks in one GPU's memory the same knowledge
// lets the quantiser place each row at its final grouped position.
// moe_combine_partial: the combine with send-side reduction in one pass --
//   per token, the partial row of each expert rank is formed from y, written
//   to its place, and added into the output.
// moe_dispatch_signalled: k_route, then the send and the receive shuffle as
//   two groups of CTAs of one co-resident kernel, handing rows over by
//   per-(sender, receiver) arrival flags.
#include <cstdint>

#include "launch.h"
#include "moeroute.h"
#include "trace.h"

namespace {

bool aligned(const void *p, long long bytes) {
    return bytes == 0 || (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0);
}

}  // namespace

// The buffers moe_dispatch and moe_dispatch_send_recv touch.
static int check_dispatch(const moe_shape *sh, const moe_buffers *b, moe_sizes &z) {
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!b) return MOE_EINVAL;
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
    return MOE_OK;
}

extern "C" int moe_dispatch_send_recv(const moe_shape *sh, const moe_buffers *b, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_dispatch(sh, b, z);
    if (rc != MOE_OK) return rc;
    if (moe::launch_dispatch_fused(*sh, (int)z.cap, b->x, b->topk_idx, b->slot_row,
                                   b->expert_send_off, b->seg_off, b->send_q, b->send_s,
                                   b->send_tok, b->grp_q, b->grp_s, b->grp_src, b->status,
                                   reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

extern "C" int moe_dispatch(const moe_shape *sh, const moe_buffers *b, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_dispatch(sh, b, z);
    if (rc != MOE_OK) return rc;
    if (moe::launch_route(*sh, (int)z.cap, b->topk_idx, b->expert_count, b->send_off,
                          b->expert_send_off, b->slot_row, b->grp_off, b->seg_off, b->csend_off,
                          b->m_sizes, b->status, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return MOE_ECUDA;
    // the dispatch may start while the routing kernel runs (it waits for the
    // routing outputs on the device)
    if (moe::launch_dispatch_fused(*sh, (int)z.cap, b->x, b->topk_idx, b->slot_row,
                                   b->expert_send_off, b->seg_off, b->send_q, b->send_s,
                                   b->send_tok, b->grp_q, b->grp_s, b->grp_src, b->status,
                                   reinterpret_cast<cudaStream_t>(stream), true) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

extern "C" int moe_dispatch_signalled(const moe_shape *sh, const moe_buffers *b, int32_t *sig,
                                      void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_dispatch(sh, b, z);
    if (rc != MOE_OK) return rc;
    if (!aligned(sig, z.bytes_sig)) return MOE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (moe::launch_route(*sh, (int)z.cap, b->topk_idx, b->expert_count, b->send_off,
                          b->expert_send_off, b->slot_row, b->grp_off, b->seg_off, b->csend_off,
                          b->m_sizes, b->status, st) != cudaSuccess)
        return MOE_ECUDA;
    if (moe::launch_dispatch_signalled(*sh, (int)z.cap, b->x, b->topk_idx, b->slot_row,
                                       b->send_off, b->expert_send_off, b->seg_off, b->send_q,
                                       b->send_s, b->send_tok, b->grp_q, b->grp_s, b->grp_src, sig,
                                       b->status, st) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

extern "C" int moe_combine(const moe_shape *sh, const moe_buffers *b, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!b) return MOE_EINVAL;
    if (!aligned(b->topk_idx, z.bytes_topk_idx) || !aligned(b->topk_w, z.bytes_topk_idx) ||
        !aligned(b->y, z.bytes_y) || !aligned(b->expert_send_off, z.bytes_expert_send_off) ||
        !aligned(b->send_off, z.bytes_send_off) || !aligned(b->slot_row, z.bytes_topk_idx) ||
        !aligned(b->seg_off, z.bytes_seg_off) || !aligned(b->csend_off, z.bytes_send_off) ||
        !aligned(b->csend, z.bytes_y) || !aligned(b->out, z.bytes_x) || !aligned(b->status, 4))
        return MOE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (moe::launch_combine_fused(*sh, (int)z.cap, b->y, b->topk_idx, b->topk_w, b->slot_row,
                                  b->expert_send_off, b->seg_off, b->send_off, b->csend_off,
                                  b->csend, b->out, st) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

extern "C" int moe_combine_partial(const moe_shape *sh, const moe_buffers *b, uint16_t *part,
                                   void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!b) return MOE_EINVAL;
    if (!aligned(b->topk_idx, z.bytes_topk_idx) || !aligned(b->topk_w, z.bytes_topk_idx) ||
        !aligned(b->y, z.bytes_y) || !aligned(b->expert_send_off, z.bytes_expert_send_off) ||
        !aligned(b->slot_row, z.bytes_topk_idx) || !aligned(b->seg_off, z.bytes_seg_off) ||
        !aligned(b->out, z.bytes_x) || !aligned(part, z.bytes_part))
        return MOE_EINVAL;
    if (moe::launch_combine_partial(*sh, (int)z.cap, b->y, b->topk_idx, b->topk_w, b->slot_row,
                                    b->expert_send_off, b->seg_off, part, b->out,
                                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}
