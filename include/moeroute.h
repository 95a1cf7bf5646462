/*
 * moeroute.h -- C ABI of libmoeroute: MoE expert-parallel dispatch and
 * combine for one GB300 (sm_103a), with the N expert-parallel ranks held as N
 * slices of the one GPU's memory.
 *
 * The operations follow "Enabling trillion-parameter models on AWS EFA"
 * (Perplexity blog):
 *   - Introduction: dispatch splits each rank's tokens and sends each to the
 *     ranks that host its experts; combine brings the expert outputs back and
 *     takes each token's weighted average.
 *   - "EFA-based MoE all-to-all": both are split into a send half and a
 *     receive half so other work can run in between.
 *   - "Send and receive buffers": per-expert token counts are exchanged first
 *     so that every sender can lay out its writes contiguously per peer and
 *     every receiver knows where each sender's tokens land; a rank receives
 *     at most N*T*max(R, E/N) tokens.
 *   - "Dispatch and combine": counting with shared-memory atomics in one
 *     block, a cumulative sum to offsets, packing into contiguous per-peer
 *     send buffers, receive-side offsets once all routing info is in, the
 *     shuffle into the grouped-GEMM input, and a combine that packs outputs
 *     per peer and accumulates the weighted average on the receiving side.
 *   - "Evaluation: dispatch/combine latency": block-scaled fp8 dispatch and
 *     bf16 combine.
 *
 * Notation: N ranks, T tokens per rank, E experts, R experts per token
 * (top-k), H hidden size.  Er = E/N experts per rank; expert e lives on rank
 * e / Er.  Sb = H/128 scale blocks per row.  cap = grouped rows per rank.
 *
 * Layout: every per-rank array is a slab [N][...] in one allocation; rank
 * r's slice starts at r * (slice size).  All arrays are row-major and dense.
 *   topk_idx        int32 [N][T][R]     expert ids chosen by the router
 *   topk_w          float [N][T][R]     their combine weights
 *   x               bf16  [N][T][H]     token activations (raw bf16 bits)
 *   expert_count    int32 [N][E]        tokens rank s sends to expert e
 *   send_off        int32 [N][N+1]      exclusive scan over peers
 *   expert_send_off int32 [N][E+1]      exclusive scan over experts
 *   slot_row        int32 [N][T][R]     send-buffer row of each assignment
 *                                       (-1: expert id outside [0, E))
 *   send_q          u8    [N][T*R][H]   fp8 e4m3 payload, per-peer contiguous
 *   send_s          float [N][T*R][Sb]  per-block scales of each send row
 *   send_tok        int32 [N][T*R]      source token of each send row
 *   grp_off         int32 [N][Er+1]     first grouped row of each local
 *                                       expert; grp_off[r][Er] = rows received
 *   seg_off         int32 [N][Er][N]    grouped row where sender s's run of
 *                                       local expert j starts
 *   csend_off       int32 [N][N+1]      row in the combine send buffer where
 *                                       the rows going back to s start
 *   m_sizes         int32 [N][Er]       rows per local expert (GEMM sizes)
 *   grp_q           u8    [N][cap][H]   grouped fp8 payload (GEMM input)
 *   grp_s           float [N][cap][Sb]  grouped scales
 *   grp_src         int32 [N][cap][2]   (source rank, source token) per row
 *   y               bf16  [N][cap][H]   expert outputs, grouped layout
 *   csend           bf16  [N][cap][H]   combine send buffer, per-destination
 *                                       contiguous
 *   out             bf16  [N][T][H]     combined output
 *
 * Ownership: every pointer is device memory owned by the caller (sized with
 * moe_sizes_query), except that x and out may also be pinned host memory
 * (cudaHostAlloc / page-locked): the kernels then read x and write out
 * directly over the CPU-GPU link, with no separate copy.  The library
 * allocates nothing and keeps no state between calls, apart from the fixed
 * static scratch array that moe_dispatch_signalled_static uses instead of a
 * caller buffer (see there) and host-side caches of launch properties per
 * device (SM count, occupancy, cluster limits; filled on a device's first
 * call, under a lock, so host threads may call at once, each with its own
 * buffers).  `stream` is a cudaStream_t (NULL = legacy default stream).
 *
 * Execution: calls only enqueue work on `stream` and never wait for the
 * device; sequences of the calls other than moe_dispatch_signalled_static can
 * be captured in a CUDA graph (tested).  Order on the stream replaces the
 * pages' receive-side waits and barriers.
 *
 * Errors: argument checks run on the host before anything is enqueued and
 * return MOE_EINVAL; a failed launch returns MOE_ECUDA.  Faults found on the
 * device are OR-ed into the int32 at `status` (device memory), which
 * moe_route_count clears first; read it after the stream has finished.  No
 * kernel traps, asserts or waits without a bound.
 */
#ifndef MOEROUTE_H
#define MOEROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_EINVAL (-1)     /* bad shape, null or misaligned pointer */
#define MOE_ENOTSUP (-2)    /* shape outside the supported limits below */
#define MOE_ECUDA (-3)      /* a CUDA call or launch failed */

#define MOE_ST_BAD_EXPERT 1 /* an expert id was outside [0, E): assignment skipped */
#define MOE_ST_CAPACITY 2   /* a rank received more than cap rows: extra rows dropped */
#define MOE_ST_TIMEOUT 4    /* a bounded wait inside a kernel gave up */

/* Supported limits (MOE_ENOTSUP beyond them): 1 <= N <= E <= 1024, E % N == 0,
 * 1 <= R <= min(E, 32), 0 <= T, T*R < 2^31, 128 <= H <= 65536 with
 * H % 128 == 0, N*cap < 2^31. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

typedef struct {
    int N;   /* ranks */
    int T;   /* tokens per rank */
    int E;   /* experts */
    int R;   /* experts per token */
    int H;   /* hidden size, multiple of 128 */
    int cap; /* grouped rows per rank; 0 selects N*T*min(R, E/N), which holds
                every routing whose R experts per token are distinct */
} moe_shape;

/* Byte sizes of every buffer for a shape (whole slab, all N ranks). */
typedef struct {
    int64_t cap;            /* effective grouped rows per rank */
    int64_t send_rows;      /* T*R rows per rank */
    int64_t bytes_x;        /* also bytes_out */
    int64_t bytes_topk_idx; /* also topk_w, slot_row */
    int64_t bytes_expert_count;
    int64_t bytes_send_off; /* also csend_off */
    int64_t bytes_expert_send_off;
    int64_t bytes_grp_off;
    int64_t bytes_seg_off;
    int64_t bytes_m_sizes;
    int64_t bytes_send_q;
    int64_t bytes_send_s;
    int64_t bytes_send_tok;
    int64_t bytes_grp_q;
    int64_t bytes_grp_s;
    int64_t bytes_grp_src;
    int64_t bytes_y;        /* also bytes_csend */
    /* low-latency layout (moe_dispatch_ll): a T-row region per (receiver,
     * local expert, sender), N*E*T rows in all */
    int64_t ll_rows;
    int64_t bytes_ll_q;     /* ll_rows * H (fp8) */
    int64_t bytes_ll_s;     /* ll_rows * H/128 * 4 */
    int64_t bytes_ll_src;   /* ll_rows * 4 */
    int64_t bytes_ll_count; /* N*E*4: [N][Er][N] */
    int64_t bytes_ll_y;     /* ll_rows * H * 2 (bf16 expert outputs) */
    int64_t bytes_sig;      /* (2*N*N + 4) * 4: moe_dispatch_signalled's flags */
    int64_t bytes_part;     /* N*N*T*H * 2: send-side-reduction partial rows */
} moe_sizes;

/* Fill *out for *shape.  Host only.  MOE_EINVAL / MOE_ENOTSUP on a bad shape. */
int moe_sizes_query(const moe_shape *shape, moe_sizes *out);

/* Dispatch send, step 1 ("Dispatch and combine": per-expert counts in one
 * block per rank -- shared-memory atomics on the page, per-warp shared-memory
 * tables here, with the same counts -- then a cumulative sum).
 * Clears *status.  One thread block per rank s:
 *   expert_count[s][e]   = #{(t,k): topk_idx[s][t][k] == e}
 *   expert_send_off[s][] = exclusive scan of expert_count[s][] (E+1 entries)
 *   send_off[s][p]       = expert_send_off[s][p*Er]  (N+1 entries)
 *   slot_row[s][t][k]    = expert_send_off[s][e] + number of earlier (t',k')
 *                          of rank s, in flattened order t'*R+k', with the
 *                          same expert; -1 (and MOE_ST_BAD_EXPERT) when the id
 *                          is outside [0, E). */
int moe_route_count(const moe_shape *shape, const int32_t *topk_idx, int32_t *expert_count,
                    int32_t *send_off, int32_t *expert_send_off, int32_t *slot_row,
                    int32_t *status, void *stream);

/* Routing-information exchange and receive-side offsets ("Send and receive
 * buffers"; "Dispatch and combine": once a rank has everyone's routing info
 * it computes the offsets for dispatch and combine).  For receiver r and its
 * local expert j (e = r*Er + j), with the runs ordered by j then sender s:
 *   seg_off[r][j][s] = sum of expert_count[s'][e'] over all runs before (j, s)
 *   grp_off[r][j]    = seg_off[r][j][0];  grp_off[r][Er] = rows r receives
 *   m_sizes[r][j]    = sum_s expert_count[s][e]
 *   csend_off[r][s]  = sum_{s' < s} (send_off[s'][r+1] - send_off[s'][r])
 * Sets MOE_ST_CAPACITY when some rank receives more than cap rows. */
int moe_exchange(const moe_shape *shape, const int32_t *expert_count, const int32_t *send_off,
                 int32_t *grp_off, int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes,
                 int32_t *status, void *stream);

/* moe_route_count and moe_exchange in one launch (same outputs, same status
 * bits, *status cleared first).  Block r plays sender r, as in
 * moe_route_count, and receiver r, as in moe_exchange; instead of waiting for
 * the other senders' counts it recounts, from all ranks' topk_idx, the
 * assignments that land on its own experts.  The pages exchange counts
 * between ranks first ("Send and receive buffers"); on one GPU every rank's
 * ids are already in memory, so no rank has to wait for another. */
int moe_route(const moe_shape *shape, const int32_t *topk_idx, int32_t *expert_count,
              int32_t *send_off, int32_t *expert_send_off, int32_t *slot_row, int32_t *grp_off,
              int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes, int32_t *status,
              void *stream);

/* Dispatch send, step 2: block-scaled fp8 quantisation fused with the pack
 * ("Dispatch and combine"; "Evaluation": block-scaled fp8 dispatch).  Per
 * token and 128-element block: amax = max|x|, scale = amax/448 (fp32
 * division), q = e4m3 round-to-nearest-even with saturation of x/scale (fp32
 * division); amax == 0 gives scale 0 and zero bytes.  The token's payload,
 * scales and id go to send rows slot_row[s][t][k] for every k with a valid
 * slot.  Rows of send_q no assignment maps to are left untouched. */
int moe_dispatch_send(const moe_shape *shape, const uint16_t *x_bf16, const int32_t *slot_row,
                      uint8_t *send_q, float *send_s, int32_t *send_tok, int32_t *status,
                      void *stream);

/* Dispatch receive: shuffle into the expert-grouped layout handed to the
 * grouped GEMM ("Dispatch and combine": tokens are shuffled from the receive
 * buffer into the grouped-GEMM input).  For every receiver r, local expert j
 * and sender s, the run of expert_count[s][e] rows that s packed for e
 * (from send row expert_send_off[s][e]) is copied to grouped rows from
 * seg_off[r][j][s], with its scales; grp_src gets (s, source token).  The
 * exchange is a device-side pull from the sender's slice.  Rows at or beyond
 * cap are dropped (MOE_ST_CAPACITY was set by moe_exchange).  Rows >= the
 * received count are left untouched. */
int moe_dispatch_recv(const moe_shape *shape, const uint8_t *send_q, const float *send_s,
                      const int32_t *send_tok, const int32_t *expert_count,
                      const int32_t *expert_send_off, const int32_t *seg_off, uint8_t *grp_q,
                      float *grp_s, int32_t *grp_src, int32_t *status, void *stream);

/* Combine send: expert rank r copies each run of outputs (grouped rows from
 * seg_off[r][j][s]) into its combine send buffer at
 *   csend_off[r][s] + (expert_send_off[s][e] - send_off[s][r])
 * so the rows going back to s are contiguous and in s's own send order ("one
 * write per peer").  A row whose grouped position was dropped is sent as
 * zeros; a row at or beyond cap in csend is dropped. */
int moe_combine_send(const moe_shape *shape, const uint16_t *y_bf16, const int32_t *expert_count,
                     const int32_t *expert_send_off, const int32_t *send_off,
                     const int32_t *seg_off, const int32_t *csend_off, uint16_t *csend,
                     int32_t *status, void *stream);

/* Combine receive: weighted average accumulated on the receiving side
 * ("Dispatch and combine"; the evaluation notes this receive-side-only
 * accumulation).  For token t of rank s:
 *   acc = 0; for k = 0..R-1: acc = fmaf(topk_w[s][t][k], row_k, acc)
 *   out[s][t] = bf16 round-to-nearest-even(acc)
 * row_k is read from rank p = e/Er's combine send buffer at
 *   csend_off[p][s] + (slot_row[s][t][k] - send_off[s][p]).
 * Skipped (invalid id) and dropped (>= cap) assignments contribute nothing. */
int moe_combine_recv(const moe_shape *shape, const uint16_t *csend, const int32_t *topk_idx,
                     const float *topk_w, const int32_t *slot_row, const int32_t *send_off,
                     const int32_t *csend_off, uint16_t *out_bf16, int32_t *status,
                     void *stream);

/* Stand-in for the grouped GEMM between dispatch and combine (the pages'
 * expert computation is out of scope here):
 *   y = bf16_rn((e4m3_decode(q) * scale) * s_e),  fp32 multiplies,
 * s_e = 1 for mode 0 (identity) and 2^((e mod 3) - 1) for mode 1 (a fixed
 * per-expert scale).  Writes the received rows of every rank; other rows of
 * y are left untouched. */
int moe_expert_standin(const moe_shape *shape, int mode, const uint8_t *grp_q,
                       const float *grp_s, const int32_t *grp_off, uint16_t *y_bf16,
                       void *stream);

/* The fp32 -> e4m3 conversion the quantiser applies (round to nearest even,
 * saturate to +-448), element-wise over n values; exposed so the encoder can
 * be compared with other implementations. */
int moe_e4m3_encode(const float *v, uint8_t *out, int64_t n, void *stream);

/* ---------------------------------------------------------------- fused
 * The whole dispatch and the whole combine as one call each, with the same
 * outputs, bit for bit, as the separate calls above.  They differ in how the
 * bytes move: moe_dispatch quantises each token once and writes its fp8 rows
 * to the send buffer and to their grouped rows in the same pass (the receive
 * shuffle never re-reads the send buffer); moe_combine reads each expert
 * output row once, writes it to its combine send row and accumulates it into
 * the token's output in the same pass (the combine send buffer is written but
 * not read back).  On the pages each sender learns the receivers' offsets
 * from the routing exchange and writes its tokens straight to their places
 * ("Send and receive buffers"); with every rank in one GPU's memory that
 * knowledge lets the quantiser place each row at its final position. */
typedef struct {
    const int32_t *topk_idx;   /* [N][T][R] */
    const float *topk_w;       /* [N][T][R] (combine) */
    const uint16_t *x;         /* [N][T][H] bf16 (dispatch) */
    int32_t *expert_count;     /* [N][E] */
    int32_t *send_off;         /* [N][N+1] */
    int32_t *expert_send_off;  /* [N][E+1] */
    int32_t *slot_row;         /* [N][T][R] */
    int32_t *grp_off;          /* [N][Er+1] */
    int32_t *seg_off;          /* [N][Er][N] */
    int32_t *csend_off;        /* [N][N+1] */
    int32_t *m_sizes;          /* [N][Er] */
    uint8_t *send_q;           /* [N][T*R][H] */
    float *send_s;             /* [N][T*R][H/128] */
    int32_t *send_tok;         /* [N][T*R] */
    uint8_t *grp_q;            /* [N][cap][H] */
    float *grp_s;              /* [N][cap][H/128] */
    int32_t *grp_src;          /* [N][cap][2] */
    const uint16_t *y;         /* [N][cap][H] bf16 expert outputs (combine) */
    uint16_t *csend;           /* [N][cap][H] */
    uint16_t *out;             /* [N][T][H] bf16 (combine) */
    int32_t *status;           /* one int32 */
} moe_buffers;

/* moe_dispatch_send and moe_dispatch_recv in one kernel, given the routing
 * arrays of a moe_route (or moe_route_count + moe_exchange) of the same
 * topk_idx: each token is quantised once and its fp8 rows, scales and ids go
 * to the send buffer and to their grouped rows.  Does not clear *status. */
int moe_dispatch_send_recv(const moe_shape *shape, const moe_buffers *b, void *stream);

/* moe_route, then moe_dispatch_send_recv.  Uses x,
 * topk_idx, the routing arrays, the send buffers and the grouped buffers;
 * *status is cleared first.  Outputs: everything moe_route_count,
 * moe_exchange, moe_dispatch_send and moe_dispatch_recv write.  The
 * dispatch kernel is launched as the routing kernel's programmatic
 * dependent: it starts loading x while the routing kernel runs and waits on
 * the device for its outputs (x must therefore be complete when the call is
 * made, as for every other call; the stream order before the call is kept). */
int moe_dispatch(const moe_shape *shape, const moe_buffers *b, void *stream);

/* moe_combine_send + moe_combine_recv in one kernel.  Uses y, topk_idx,
 * topk_w, the routing arrays (from a dispatch of the same topk_idx), csend
 * and out.  Outputs: csend and out, as the two separate calls write them. */
int moe_combine(const moe_shape *shape, const moe_buffers *b, void *stream);

/* ---------------------------------------------------------------- send-side reduction
 * The combine with send-side accumulation, the alternative the EFA page's
 * evaluation ("Evaluation: dispatch/combine latency", prefill) contrasts with
 * its receive-side-only accumulation: summing on the sending side cuts the
 * bytes sent, with some risk to accuracy.  On expert rank r, for each token t
 * of each rank s with at least one expert on r, the weighted outputs of those
 * experts are summed (fp32 fused multiply-add in slot order; an output whose
 * grouped row was dropped at capacity counts as zero) and rounded once to
 * bf16:
 *   part     bf16  [N][N][T][H]   row (r, s, t); rows of an (r, s, t) without
 *                                 an expert of r are left untouched
 * The receiver adds its token's partial rows in ascending rank order in fp32
 * and rounds once to bf16 (0 for a token without valid experts).  Against
 * the exact weighted sum X: |out - X| <= 2^-7 * sum_k |w_k y_k| (one bf16
 * rounding per partial and one at the end) -- a different result from
 * moe_combine_recv, whose one rounding gives |out - X| <= 2^-8 |X| + fp32
 * error.  Bytes sent: one row per (token, expert rank) instead of one per
 * (token, expert).  Host errors as above; no status bits. */

/* Sending side: writes the partial rows.  y, topk_idx, topk_w, slot_row,
 * expert_send_off, seg_off as for moe_combine_send / moe_combine_recv. */
int moe_combine_partial_send(const moe_shape *shape, const uint16_t *y_bf16,
                             const int32_t *topk_idx, const float *topk_w,
                             const int32_t *slot_row, const int32_t *expert_send_off,
                             const int32_t *seg_off, uint16_t *part, void *stream);

/* Receiving side: out[s][t] = bf16_rn(sum over ranks r of the token's experts,
 * ascending, of part[r][s][t]).  out may be pinned host memory. */
int moe_combine_partial_recv(const moe_shape *shape, const uint16_t *part,
                             const int32_t *topk_idx, const int32_t *slot_row,
                             uint16_t *out_bf16, void *stream);

/* Both in one pass: each partial row is formed once, written to part and
 * added into out.  Uses y, topk_idx, topk_w, slot_row, expert_send_off,
 * seg_off and out of *b. */
int moe_combine_partial(const moe_shape *shape, const moe_buffers *b, uint16_t *part,
                        void *stream);

/* ---------------------------------------------------------------- signalled
 * moe_route, then the dispatch send and the dispatch receive shuffle in ONE
 * kernel whose parts hand rows over by per-group arrival flags rather than
 * by a kernel boundary: the one-GPU form of the decoupled signalling of "MoE
 * multi-node inference bottleneck overturned: Perseus removes hidden
 * serialization" (section 3, Algorithm 1, Figure 6 -- transfers first, then
 * one fence and one signal per destination group, set by whichever
 * participant completes the group).  Packing CTAs quantise and write the
 * send rows exactly as moe_dispatch_send; each (sender s, receiver r) group
 * is the run of s's send buffer bound for r (send_off[s][r] ..
 * send_off[s][r+1]).  Every row written adds one to the group's counter
 * after a CTA barrier and a release fence that order the row's stores
 * before it; the writer that completes the group sets its flag.  Receiving CTAs copy each send row to
 * its grouped row exactly as moe_dispatch_recv, once the row's group flag is
 * set, so a receiver starts on sender s while later senders are still being
 * packed.  Outputs: everything moe_dispatch writes, bit for bit.
 *
 * sig: int32 scratch of bytes_sig bytes, caller-owned device memory, 16-byte
 *   aligned: [N][N] group counters, [N][N] group flags, one completion
 *   counter.  It must be all zero before the first call; every call leaves it
 *   zero again (the kernel's last CTA clears it).  Calls that share one sig
 *   must not overlap in time (the same stream orders them).
 * Every CTA of the kernel is resident at once (a cooperative launch; it
 * fails with MOE_ECUDA rather than run partly resident).  Each wait is
 * bounded (about a second); a group that never completes (a sig that was not
 * zero) sets MOE_ST_TIMEOUT, its rows are not copied, and the call still
 * returns and clears sig.  *status is cleared first. */
int moe_dispatch_signalled(const moe_shape *shape, const moe_buffers *b, int32_t *sig,
                           void *stream);

/* ---------------------------------------------------------------- no allocation
 * moe_dispatch_signalled with its flag scratch in a static device array of
 * this library instead of the caller's sig buffer; the pages have no
 * counterpart (it is an interface convenience, not a step of the method).
 * It is for callers that cannot allocate the extra scratch: a serving
 * process that carves device memory into its own arenas at start-up and
 * must not allocate while serving, or a C caller that holds only the
 * moe_buffers set another framework allocated.  The call itself allocates
 * nothing (no cudaMalloc, no allocating library routine).
 * Limit: N <= MOE_SIG_STATIC_MAX_N; a larger N returns MOE_ENOTSUP before any
 * CUDA call.  The first call with a given device current looks up the
 * array's address on that device (cudaGetSymbolAddress) -- make that first
 * call before any stream capture.  Each call clears the scratch it uses
 * (cudaMemsetAsync on `stream`), then does exactly what moe_dispatch_signalled
 * does.  All calls on one device share the array: calls that overlap in time
 * (several streams or host threads) race and give wrong results; order them
 * on one stream. */
#define MOE_SIG_STATIC_MAX_N 64
int moe_dispatch_signalled_static(const moe_shape *shape, const moe_buffers *b, void *stream);

/* ---------------------------------------------------------------- low latency
 * Dispatch and combine in one kernel each, for decode-sized batches: the
 * low-latency mode of the RoCE->EFA page (section 4.4) presets a per-rank
 * token limit and preallocates fixed receive buffers, so no count-then-
 * allocate round is needed and the whole dispatch is one kernel that a CUDA
 * graph can capture.  Here receiver r keeps a T-row region for each local
 * expert j and sender s:
 *   ll_q     u8    [N][Er][N][T][H]   row ((r*Er + j)*N + s)*T + u
 *   ll_s     float [N][Er][N][T][H/128]
 *   ll_src   int32 [N][Er][N][T]      source token t of each row
 *   ll_count int32 [N][Er][N]         rows in each region (may exceed T:
 *                                     the rest are dropped, MOE_ST_CAPACITY)
 *   ll_row   int32 [N][T][R]          row of each assignment, -1 if none
 *   y_ll     bf16  [N][Er][N][T][H]   expert outputs in the same rows
 * where u is the assignment's stable rank among sender s's assignments to
 * expert e = r*Er + j (the order of slot_row).  No routing exchange, send
 * buffer or combine send buffer is used: every row's position follows from
 * the sender's own ids.  Rows past ll_count are left untouched.  Limits: T <=
 * 1024 (MOE_ENOTSUP beyond), N*E*T < 2^31. */

/* Quantise every token (as moe_dispatch_send) and place its rows, scales and
 * token id in the low-latency layout; writes ll_row and ll_count (all zero
 * for an empty batch).  Clears *status first; MOE_ST_BAD_EXPERT / MOE_ST_CAPACITY as for the main path.
 * One kernel: with at most 2048 ids per rank each token's rows come from a
 * count of the sender's earlier ids; longer batches rank every sender's ids
 * once in the same (co-resident) launch first.  The outputs are the same. */
int moe_dispatch_ll(const moe_shape *shape, const uint16_t *x_bf16, const int32_t *topk_idx,
                    uint8_t *ll_q, float *ll_s, int32_t *ll_src, int32_t *ll_count,
                    int32_t *ll_row, int32_t *status, void *stream);

/* The grouped-GEMM stand-in of moe_expert_standin over the low-latency
 * layout (rows u < min(ll_count, T) of each region). */
int moe_expert_standin_ll(const moe_shape *shape, int mode, const uint8_t *ll_q,
                          const float *ll_s, const int32_t *ll_count, uint16_t *y_ll,
                          void *stream);

/* Weighted average of each token's rows y_ll[ll_row[s][t][k]], fp32 FMA in
 * slot order, one bf16 rounding (as moe_combine_recv).  out may be pinned host
 * memory. */
int moe_combine_ll(const moe_shape *shape, const uint16_t *y_ll, const float *topk_w,
                   const int32_t *ll_row, uint16_t *out_bf16, int32_t *status, void *stream);

/* Static description of an error code or status bit set. */
const char *moe_strerror(int code);

/* Library version, (major << 16) | minor. */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEROUTE_H */
