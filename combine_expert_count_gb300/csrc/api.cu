// api.cu -- the extern "C" boundary of libmoeroute: argument validation on
// the host, then asynchronous launches on the caller's stream.  Nothing here
// allocates device memory, synchronises the host or keeps state between
// calls, except per-device caches of launch properties (SM count here,
// occupancies and cluster limits beside each launcher).
#include <atomic>
#include <cstdint>
#include <cstring>

#include "launch.h"
#include "moeroute.h"
#include "trace.h"

namespace moe {

int sm_count() {
    static std::atomic<int> cached[64];  // zero-initialised: not yet asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace moe

namespace {

int check_shape(const moe_shape *sh) {
    if (!sh) return MOE_EINVAL;
    if (sh->N <= 0 || sh->T < 0 || sh->E <= 0 || sh->R <= 0 || sh->H <= 0 || sh->cap < 0)
        return MOE_EINVAL;
    if (sh->H % 128 != 0 || sh->E % sh->N != 0 || sh->R > sh->E) return MOE_EINVAL;
    if (sh->E > MOE_MAX_EXPERTS || sh->R > MOE_MAX_TOPK || sh->H > 65536) return MOE_ENOTSUP;
    if ((int64_t)sh->T * sh->R >= ((int64_t)1 << 31)) return MOE_ENOTSUP;
    return MOE_OK;
}

int64_t eff_cap(const moe_shape *sh) {
    if (sh->cap > 0) return sh->cap;
    const int64_t Er = sh->E / sh->N;
    return (int64_t)sh->N * sh->T * (sh->R < Er ? sh->R : Er);
}

// Effective cap, or a negative error code.
int shape_cap(const moe_shape *sh, int *cap) {
    int rc = check_shape(sh);
    if (rc != MOE_OK) return rc;
    const int64_t c = eff_cap(sh);
    if ((int64_t)sh->N * c >= ((int64_t)1 << 31)) return MOE_ENOTSUP;
    *cap = (int)c;
    return MOE_OK;
}

// A pointer may be null only when the buffer it names is empty.
bool ok_ptr(const void *p, int64_t bytes) {
    if (bytes == 0) return true;
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ECUDA; }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

int moe_version(void) { return (1 << 16) | 0; }

const char *moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_EINVAL: return "invalid argument (shape, null or misaligned pointer)";
        case MOE_ENOTSUP: return "shape outside the supported limits";
        case MOE_ECUDA: return "CUDA launch or call failed";
        case MOE_ST_BAD_EXPERT: return "device status: expert id outside [0, E), assignment skipped";
        case MOE_ST_CAPACITY: return "device status: a rank received more than cap rows, extra rows dropped";
        case MOE_ST_TIMEOUT: return "device status: a bounded wait gave up";
        default: return "unknown code or several status bits";
    }
}

int moe_sizes_query(const moe_shape *sh, moe_sizes *out) {
    int cap = 0;
    int rc = shape_cap(sh, &cap);
    if (rc != MOE_OK) return rc;
    if (!out) return MOE_EINVAL;
    const int64_t N = sh->N, T = sh->T, E = sh->E, R = sh->R, H = sh->H, Er = E / N,
                  Sb = H / 128;
    std::memset(out, 0, sizeof(*out));
    out->cap = cap;
    out->send_rows = T * R;
    out->bytes_x = N * T * H * 2;
    out->bytes_topk_idx = N * T * R * 4;
    out->bytes_expert_count = N * E * 4;
    out->bytes_send_off = N * (N + 1) * 4;
    out->bytes_expert_send_off = N * (E + 1) * 4;
    out->bytes_grp_off = N * (Er + 1) * 4;
    out->bytes_seg_off = N * Er * N * 4;
    out->bytes_m_sizes = N * Er * 4;
    out->bytes_send_q = N * T * R * H;
    out->bytes_send_s = N * T * R * Sb * 4;
    out->bytes_send_tok = N * T * R * 4;
    out->bytes_grp_q = N * (int64_t)cap * H;
    out->bytes_grp_s = N * (int64_t)cap * Sb * 4;
    out->bytes_grp_src = N * (int64_t)cap * 8;
    out->bytes_y = N * (int64_t)cap * H * 2;
    out->ll_rows = N * E * T;
    out->bytes_ll_q = out->ll_rows * H;
    out->bytes_ll_s = out->ll_rows * Sb * 4;
    out->bytes_ll_src = out->ll_rows * 4;
    out->bytes_ll_count = N * E * 4;
    out->bytes_ll_y = out->ll_rows * H * 2;
    out->bytes_sig = (2 * N * N + 4) * 4;
    out->bytes_part = N * N * T * H * 2;
    return MOE_OK;
}

// The low-latency calls' extra limits.
static int check_ll(const moe_shape *sh, moe_sizes *z) {
    int rc = moe_sizes_query(sh, z);
    if (rc != MOE_OK) return rc;
    if (sh->T > 1024 || z->ll_rows >= ((int64_t)1 << 31)) return MOE_ENOTSUP;
    return MOE_OK;
}

int moe_route_count(const moe_shape *sh, const int32_t *topk_idx, int32_t *expert_count,
                    int32_t *send_off, int32_t *expert_send_off, int32_t *slot_row,
                    int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(topk_idx, z.bytes_topk_idx) || !ok_ptr(slot_row, z.bytes_topk_idx) ||
        !ok_ptr(expert_count, z.bytes_expert_count) || !ok_ptr(send_off, z.bytes_send_off) ||
        !ok_ptr(expert_send_off, z.bytes_expert_send_off) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_route_count(*sh, topk_idx, expert_count, send_off,
                                           expert_send_off, slot_row, status, as_stream(stream)));
}

int moe_exchange(const moe_shape *sh, const int32_t *expert_count, const int32_t *send_off,
                 int32_t *grp_off, int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes,
                 int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(expert_count, z.bytes_expert_count) || !ok_ptr(send_off, z.bytes_send_off) ||
        !ok_ptr(grp_off, z.bytes_grp_off) || !ok_ptr(seg_off, z.bytes_seg_off) ||
        !ok_ptr(csend_off, z.bytes_send_off) || !ok_ptr(m_sizes, z.bytes_m_sizes) ||
        !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_exchange(*sh, (int)z.cap, expert_count, send_off, grp_off, seg_off,
                                        csend_off, m_sizes, status, as_stream(stream)));
}

int moe_route(const moe_shape *sh, const int32_t *topk_idx, int32_t *expert_count,
              int32_t *send_off, int32_t *expert_send_off, int32_t *slot_row, int32_t *grp_off,
              int32_t *seg_off, int32_t *csend_off, int32_t *m_sizes, int32_t *status,
              void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(topk_idx, z.bytes_topk_idx) || !ok_ptr(slot_row, z.bytes_topk_idx) ||
        !ok_ptr(expert_count, z.bytes_expert_count) || !ok_ptr(send_off, z.bytes_send_off) ||
        !ok_ptr(expert_send_off, z.bytes_expert_send_off) || !ok_ptr(grp_off, z.bytes_grp_off) ||
        !ok_ptr(seg_off, z.bytes_seg_off) || !ok_ptr(csend_off, z.bytes_send_off) ||
        !ok_ptr(m_sizes, z.bytes_m_sizes) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_route(*sh, (int)z.cap, topk_idx, expert_count, send_off,
                                     expert_send_off, slot_row, grp_off, seg_off, csend_off,
                                     m_sizes, status, as_stream(stream)));
}

int moe_dispatch_send(const moe_shape *sh, const uint16_t *x_bf16, const int32_t *slot_row,
                      uint8_t *send_q, float *send_s, int32_t *send_tok, int32_t *status,
                      void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(x_bf16, z.bytes_x) || !ok_ptr(slot_row, z.bytes_topk_idx) ||
        !ok_ptr(send_q, z.bytes_send_q) || !ok_ptr(send_s, z.bytes_send_s) ||
        !ok_ptr(send_tok, z.bytes_send_tok) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_quant_pack(*sh, x_bf16, slot_row, send_q, send_s, send_tok, status,
                                          as_stream(stream)));
}

int moe_dispatch_recv(const moe_shape *sh, const uint8_t *send_q, const float *send_s,
                      const int32_t *send_tok, const int32_t *expert_count,
                      const int32_t *expert_send_off, const int32_t *seg_off, uint8_t *grp_q,
                      float *grp_s, int32_t *grp_src, int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(send_q, z.bytes_send_q) || !ok_ptr(send_s, z.bytes_send_s) ||
        !ok_ptr(send_tok, z.bytes_send_tok) || !ok_ptr(expert_count, z.bytes_expert_count) ||
        !ok_ptr(expert_send_off, z.bytes_expert_send_off) || !ok_ptr(seg_off, z.bytes_seg_off) ||
        !ok_ptr(grp_q, z.bytes_grp_q) || !ok_ptr(grp_s, z.bytes_grp_s) ||
        !ok_ptr(grp_src, z.bytes_grp_src) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_dispatch_pull(*sh, (int)z.cap, send_q, send_s, send_tok,
                                             expert_send_off, seg_off, grp_q, grp_s, grp_src,
                                             status, as_stream(stream)));
}

int moe_combine_send(const moe_shape *sh, const uint16_t *y_bf16, const int32_t *expert_count,
                     const int32_t *expert_send_off, const int32_t *send_off,
                     const int32_t *seg_off, const int32_t *csend_off, uint16_t *csend,
                     int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(y_bf16, z.bytes_y) || !ok_ptr(expert_count, z.bytes_expert_count) ||
        !ok_ptr(expert_send_off, z.bytes_expert_send_off) || !ok_ptr(send_off, z.bytes_send_off) ||
        !ok_ptr(seg_off, z.bytes_seg_off) || !ok_ptr(csend_off, z.bytes_send_off) ||
        !ok_ptr(csend, z.bytes_y) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_combine_pack(*sh, (int)z.cap, y_bf16, expert_send_off, send_off,
                                            seg_off, csend_off, csend, status, as_stream(stream)));
}

int moe_combine_recv(const moe_shape *sh, const uint16_t *csend, const int32_t *topk_idx,
                     const float *topk_w, const int32_t *slot_row, const int32_t *send_off,
                     const int32_t *csend_off, uint16_t *out_bf16, int32_t *status,
                     void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(csend, z.bytes_y) || !ok_ptr(topk_idx, z.bytes_topk_idx) ||
        !ok_ptr(topk_w, z.bytes_topk_idx) || !ok_ptr(slot_row, z.bytes_topk_idx) ||
        !ok_ptr(send_off, z.bytes_send_off) || !ok_ptr(csend_off, z.bytes_send_off) ||
        !ok_ptr(out_bf16, z.bytes_x) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_combine_reduce(*sh, (int)z.cap, csend, topk_idx, topk_w, slot_row,
                                              send_off, csend_off, out_bf16, as_stream(stream)));
}

int moe_combine_partial_send(const moe_shape *sh, const uint16_t *y_bf16, const int32_t *topk_idx,
                             const float *topk_w, const int32_t *slot_row,
                             const int32_t *expert_send_off, const int32_t *seg_off,
                             uint16_t *part, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(y_bf16, z.bytes_y) || !ok_ptr(topk_idx, z.bytes_topk_idx) ||
        !ok_ptr(topk_w, z.bytes_topk_idx) || !ok_ptr(slot_row, z.bytes_topk_idx) ||
        !ok_ptr(expert_send_off, z.bytes_expert_send_off) || !ok_ptr(seg_off, z.bytes_seg_off) ||
        !ok_ptr(part, z.bytes_part))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_combine_partial_send(*sh, (int)z.cap, y_bf16, topk_idx, topk_w,
                                                    slot_row, expert_send_off, seg_off, part,
                                                    as_stream(stream)));
}

int moe_combine_partial_recv(const moe_shape *sh, const uint16_t *part, const int32_t *topk_idx,
                             const int32_t *slot_row, uint16_t *out_bf16, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(part, z.bytes_part) || !ok_ptr(topk_idx, z.bytes_topk_idx) ||
        !ok_ptr(slot_row, z.bytes_topk_idx) || !ok_ptr(out_bf16, z.bytes_x))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_combine_partial_recv(*sh, part, topk_idx, slot_row, out_bf16,
                                                    as_stream(stream)));
}

int moe_expert_standin(const moe_shape *sh, int mode, const uint8_t *grp_q, const float *grp_s,
                       const int32_t *grp_off, uint16_t *y_bf16, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (mode != 0 && mode != 1) return MOE_EINVAL;
    if (!ok_ptr(grp_q, z.bytes_grp_q) || !ok_ptr(grp_s, z.bytes_grp_s) ||
        !ok_ptr(grp_off, z.bytes_grp_off) || !ok_ptr(y_bf16, z.bytes_y))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_expert_standin(*sh, (int)z.cap, mode, grp_q, grp_s, grp_off, y_bf16,
                                              as_stream(stream)));
}

int moe_dispatch_ll(const moe_shape *sh, const uint16_t *x_bf16, const int32_t *topk_idx,
                    uint8_t *ll_q, float *ll_s, int32_t *ll_src, int32_t *ll_count,
                    int32_t *ll_row, int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_ll(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(x_bf16, z.bytes_x) || !ok_ptr(topk_idx, z.bytes_topk_idx) ||
        !ok_ptr(ll_q, z.bytes_ll_q) || !ok_ptr(ll_s, z.bytes_ll_s) ||
        !ok_ptr(ll_src, z.bytes_ll_src) || !ok_ptr(ll_count, z.bytes_ll_count) ||
        !ok_ptr(ll_row, z.bytes_topk_idx) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_dispatch_ll(*sh, x_bf16, topk_idx, ll_q, ll_s, ll_src, ll_count,
                                           ll_row, status, as_stream(stream)));
}

int moe_expert_standin_ll(const moe_shape *sh, int mode, const uint8_t *ll_q, const float *ll_s,
                          const int32_t *ll_count, uint16_t *y_ll, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_ll(sh, &z);
    if (rc != MOE_OK) return rc;
    if (mode != 0 && mode != 1) return MOE_EINVAL;
    if (!ok_ptr(ll_q, z.bytes_ll_q) || !ok_ptr(ll_s, z.bytes_ll_s) ||
        !ok_ptr(ll_count, z.bytes_ll_count) || !ok_ptr(y_ll, z.bytes_ll_y))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_expert_standin_ll(*sh, mode, ll_q, ll_s, ll_count, y_ll,
                                                 as_stream(stream)));
}

int moe_combine_ll(const moe_shape *sh, const uint16_t *y_ll, const float *topk_w,
                   const int32_t *ll_row, uint16_t *out_bf16, int32_t *status, void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = check_ll(sh, &z);
    if (rc != MOE_OK) return rc;
    if (!ok_ptr(y_ll, z.bytes_ll_y) || !ok_ptr(topk_w, z.bytes_topk_idx) ||
        !ok_ptr(ll_row, z.bytes_topk_idx) || !ok_ptr(out_bf16, z.bytes_x) || !ok_ptr(status, 4))
        return MOE_EINVAL;
    return cuda_rc(moe::launch_combine_ll(*sh, y_ll, topk_w, ll_row, out_bf16, as_stream(stream)));
}

int moe_e4m3_encode(const float *v, uint8_t *out, int64_t n, void *stream) {
    MOE_TRACE_CALL();
    if (n < 0) return MOE_EINVAL;
    if (n > 0 && (v == nullptr || out == nullptr)) return MOE_EINVAL;
    return cuda_rc(moe::launch_e4m3_encode(v, out, n, as_stream(stream)));
}

}  // extern "C"
