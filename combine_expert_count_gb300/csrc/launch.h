// launch.h -- internal launchers behind the C ABI (arguments already
// validated by api.cu; all pointers device memory, all calls asynchronous).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "moeroute.h"

namespace moe {

cudaError_t launch_route_count(const moe_shape &sh, const int32_t *idx, int32_t *cnt,
                               int32_t *send_off, int32_t *eso, int32_t *slot_row,
                               int32_t *status, cudaStream_t st);

cudaError_t launch_route(const moe_shape &sh, int cap, const int32_t *idx, int32_t *cnt,
                         int32_t *send_off, int32_t *eso, int32_t *slot_row, int32_t *grp_off,
                         int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes, int32_t *status,
                         cudaStream_t st);

cudaError_t launch_exchange(const moe_shape &sh, int cap, const int32_t *cnt,
                            const int32_t *send_off, int32_t *grp_off, int32_t *seg_off,
                            int32_t *csend_off, int32_t *m_sizes, int32_t *status,
                            cudaStream_t st);

cudaError_t launch_quant_pack(const moe_shape &sh, const uint16_t *x, const int32_t *slot_row,
                              uint8_t *send_q, float *send_s, int32_t *send_tok, int32_t *status,
                              cudaStream_t st);

// Quantise + pack + receive shuffle in one pass: the fp8 rows go to the send
// buffer and, at the same time, to their grouped rows (moe_dispatch).
cudaError_t launch_dispatch_fused(const moe_shape &sh, int cap, const uint16_t *x,
                                  const int32_t *idx, const int32_t *slot_row, const int32_t *eso,
                                  const int32_t *seg_off, uint8_t *send_q, float *send_s,
                                  int32_t *send_tok, uint8_t *grp_q, float *grp_s,
                                  int32_t *grp_src, int32_t *status, cudaStream_t st,
                                  bool after_route = false);

// Quantise + pack and the receive shuffle in one co-resident grid whose
// CTAs hand rows over by per-(sender, receiver) arrival flags in `sig`
// (moe_dispatch_signalled; sig: [N][N] counters, [N][N] flags, one done
// counter, all zero on entry and on return).
cudaError_t launch_dispatch_signalled(const moe_shape &sh, int cap, const uint16_t *x,
                                      const int32_t *idx, const int32_t *slot_row,
                                      const int32_t *send_off, const int32_t *eso,
                                      const int32_t *seg_off, uint8_t *send_q, float *send_s,
                                      int32_t *send_tok, uint8_t *grp_q, float *grp_s,
                                      int32_t *grp_src, int32_t *sig, int32_t *status,
                                      cudaStream_t st);

cudaError_t launch_dispatch_pull(const moe_shape &sh, int cap, const uint8_t *send_q,
                                 const float *send_s, const int32_t *send_tok,
                                 const int32_t *eso, const int32_t *seg_off, uint8_t *grp_q,
                                 float *grp_s, int32_t *grp_src, int32_t *status, cudaStream_t st,
                                 long long row0 = 0, long long row1 = -1);

cudaError_t launch_combine_pack(const moe_shape &sh, int cap, const uint16_t *y,
                                const int32_t *eso, const int32_t *send_off,
                                const int32_t *seg_off, const int32_t *csend_off, uint16_t *csend,
                                int32_t *status, cudaStream_t st, long long row0 = 0,
                                long long row1 = -1);

cudaError_t launch_combine_reduce(const moe_shape &sh, int cap, const uint16_t *csend,
                                  const int32_t *idx, const float *w, const int32_t *slot_row,
                                  const int32_t *send_off, const int32_t *csend_off,
                                  uint16_t *out, cudaStream_t st);

// Combine send + receive in one pass (moe_combine).
cudaError_t launch_combine_fused(const moe_shape &sh, int cap, const uint16_t *y,
                                 const int32_t *idx, const float *w, const int32_t *slot_row,
                                 const int32_t *eso, const int32_t *seg_off,
                                 const int32_t *send_off, const int32_t *csend_off,
                                 uint16_t *csend, uint16_t *out, cudaStream_t st);

// Combine with send-side reduction: partial rows [N][N][T][H] bf16
// (expert rank, sender, token).
cudaError_t launch_combine_partial_send(const moe_shape &sh, int cap, const uint16_t *y,
                                        const int32_t *idx, const float *w,
                                        const int32_t *slot_row, const int32_t *eso,
                                        const int32_t *seg_off, uint16_t *pbuf, cudaStream_t st);

cudaError_t launch_combine_partial_recv(const moe_shape &sh, const uint16_t *pbuf,
                                        const int32_t *idx, const int32_t *slot_row,
                                        uint16_t *out, cudaStream_t st);

cudaError_t launch_combine_partial(const moe_shape &sh, int cap, const uint16_t *y,
                                   const int32_t *idx, const float *w, const int32_t *slot_row,
                                   const int32_t *eso, const int32_t *seg_off, uint16_t *pbuf,
                                   uint16_t *out, cudaStream_t st);

cudaError_t launch_expert_standin(const moe_shape &sh, int cap, int mode, const uint8_t *grp_q,
                                  const float *grp_s, const int32_t *grp_off, uint16_t *y,
                                  cudaStream_t st);

// Low-latency layout (fixed T-row region per (local expert, sender)).
cudaError_t launch_dispatch_ll(const moe_shape &sh, const uint16_t *x, const int32_t *idx,
                               uint8_t *ll_q, float *ll_s, int32_t *ll_src, int32_t *ll_count,
                               int32_t *ll_row, int32_t *status, cudaStream_t st);

cudaError_t launch_combine_ll(const moe_shape &sh, const uint16_t *y_ll, const float *w,
                              const int32_t *ll_row, uint16_t *out, cudaStream_t st);

cudaError_t launch_expert_standin_ll(const moe_shape &sh, int mode, const uint8_t *ll_q,
                                     const float *ll_s, const int32_t *ll_count, uint16_t *y_ll,
                                     cudaStream_t st);

cudaError_t launch_e4m3_encode(const float *v, uint8_t *out, int64_t n, cudaStream_t st);

// SM count of the current device (cached per device).
int sm_count();

// Blocks per token for the kernels that give each token (or part of one) a
// block: as many as a wave of resident blocks (SMs x `occ`) holds per token,
// rounded down so that a batch filling the wave keeps one block per token,
// at most one 16-byte chunk per thread of every row, and at least `least`.
inline int token_split(long long ntok, int H, int threads, int occ, int least) {
    long long sp = (long long)sm_count() * occ / (ntok > 0 ? ntok : 1);
    const long long most = (H >> 3) / threads;
    if (sp > most) sp = most;
    if (sp < least) sp = least;
    return (int)sp;
}

// A launch property of the current device (a kernel's occupancy, a cluster
// limit) worked out by `fill` once per (device, key) and kept.  The lookup
// and `fill` run under one lock: host threads calling at once neither race
// on the table nor launch before the attribute calls another thread makes
// inside `fill` have finished.  A failed `fill` is not kept.
class LaunchMemo {
  public:
    template <class F>
    cudaError_t get(long long key, int *out, F &&fill) {
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        std::lock_guard<std::mutex> lock(mu_);
        for (const Entry &e : entries_)
            if (e.dev == dev && e.key == key) {
                *out = e.value;
                return cudaSuccess;
            }
        int v = 0;
        err = fill(&v);
        if (err != cudaSuccess) return err;
        entries_.push_back(Entry{dev, key, v});
        *out = v;
        return cudaSuccess;
    }

  private:
    struct Entry {
        int dev;
        long long key;
        int value;
    };
    std::mutex mu_;
    std::vector<Entry> entries_;
};

}  // namespace moe
