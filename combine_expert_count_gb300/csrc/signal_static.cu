// signal_static.cu -- moe_dispatch_signalled_static: the signalled dispatch
// with its flag scratch in a file-scope device array of this library
// instead of a caller-supplied buffer, so the call allocates nothing and
// asks the caller for nothing beyond moe_dispatch's buffers.
//
// It is for callers that cannot allocate device memory at the point where
// they dispatch: a serving process that splits the GPU's memory into its
// own arenas at start-up and must not call cudaMalloc while it serves (the
// call could fail under memory pressure or break the plan), or a C program
// that receives the moe_buffers set from another framework's allocator and
// has no allocator of its own for the extra flag buffer.
//
// The array holds the scratch of shapes up to MOE_SIG_STATIC_MAX_N ranks:
// 2*N*N group counters and flags plus a completion counter, 32,784 bytes.
// Its address is looked up once per device (cudaGetSymbolAddress with that
// device current) on the first call made with that device current.  Every
// call clears the part it uses on its stream before the kernel runs.  All
// calls on one device share the array, so calls that overlap in time race.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "moeroute.h"
#include "trace.h"

namespace {

constexpr int kMaxN = MOE_SIG_STATIC_MAX_N;
constexpr size_t kInts = 2 * (size_t)kMaxN * kMaxN + 4;

static __device__ __align__(256) int32_t g_sig_scratch[kInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t *g_sig_ptr[kMaxDevices];

// The array's address on the current device, looked up on first use.
int scratch_ptr(int32_t **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MOE_ENOTSUP;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sig_ptr[dev] == nullptr) {
        int32_t *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_sig_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return MOE_ECUDA;
        }
        g_sig_ptr[dev] = ptr;
    }
    *out = g_sig_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_dispatch_signalled_static(const moe_shape *sh, const moe_buffers *b,
                                             void *stream) {
    MOE_TRACE_CALL();
    moe_sizes z;
    int rc = moe_sizes_query(sh, &z);
    if (rc != MOE_OK) return rc;
    if (sh->N > kMaxN || (size_t)z.bytes_sig > kInts * sizeof(int32_t)) return MOE_ENOTSUP;
    if (b == nullptr) return MOE_EINVAL;
    int32_t *sig = nullptr;
    rc = scratch_ptr(&sig);
    if (rc != MOE_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(sig, 0, (size_t)z.bytes_sig, st) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
    }
    return moe_dispatch_signalled(sh, b, sig, stream);
}
