// rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot allocate device memory.
//
// The regular backward takes a caller-provided workspace for its per-CTA dw partial sums. Some
// callers have no way to provide one: plugins inside an inference or training engine that owns
// every device allocation and hands a plugin only its inputs and outputs, and plain C callers
// with no caching allocator, for whom a cudaMalloc and cudaFree around each call would
// synchronise the device. This entry point keeps the partial sums in a fixed array in the
// library's own device memory instead.
//
// The array is a file-scope __device__ variable of kScratchFloats floats (8 MiB): every GPU that
// loads the library holds it until the process exits. All calls on a device share it, and it
// keeps the previous call's contents; nothing in it needs to start at zero, because stage 1
// writes every element that stage 2 reads. Two calls whose kernels overlap on the GPU (on
// different streams, or from different threads without ordering) race on the array.
//
// Host code cannot use the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current) and caches it. That
// lookup is the first call's only extra work.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "launch.h"
#include "rrn.h"

namespace rrn {
namespace {

constexpr int64_t kScratchFloats = int64_t(1) << 21;  // 8 MiB of fp32 partial sums

__device__ __align__(256) float g_bwd_scratch[kScratchFloats];

constexpr int kMaxScratchDevices = 64;
std::atomic<uintptr_t> g_scratch_addr[kMaxScratchDevices];

// The scratch array's device address on the current device (looked up once per device).
int scratch_address(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return RRN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxScratchDevices) {
        const uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
        if (a) {
            *out = reinterpret_cast<float *>(a);
            return RRN_OK;
        }
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) return RRN_ERR_CUDA;
    if (dev >= 0 && dev < kMaxScratchDevices)
        g_scratch_addr[dev].store(reinterpret_cast<uintptr_t>(p), std::memory_order_release);
    *out = static_cast<float *>(p);
    return RRN_OK;
}

}  // namespace
}  // namespace rrn

extern "C" RRN_API int rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *w,
                                           const float *rstd, void *dx, float *dw, int64_t M,
                                           int64_t N, float eps, int dtype, rrn_stream_t stream) {
    using namespace rrn;
    // the regular entry point's argument checks first, so that their codes win
    int st = validate_bwd(dy, x, w, rstd, dx, dw, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) {
        // an empty sum: the regular entry point sets dw to zero and uses no workspace
        return rmsnorm_bwd(dy, x, w, rstd, dx, dw, nullptr, 0, M, N, eps, dtype, stream);
    }
    if (N > kScratchFloats) return RRN_ERR_SCRATCH;  // not even one row of partial sums fits
    // The regular plan, with the rows of partial sums stage 1 writes (one per CTA, or one per
    // cluster when a row is split over a cluster) lowered until they fit the array.
    rrn_launch cfg{};
    st = rrn_plan_bwd(dy, nullptr, x, w, dx, M, N, dtype, &cfg);
    if (st != RRN_OK) return st;
    const int64_t fit = kScratchFloats / N;
    const int per_row = cfg.cluster > 0 ? cfg.cluster : 1;  // CTAs sharing one row of sums
    if (cfg.ctas / per_row > fit) cfg.ctas = static_cast<int>(fit) * per_row;
    float *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != RRN_OK) return st;
    return rmsnorm_bwd_ex(dy, x, w, rstd, dx, dw, scratch,
                          static_cast<size_t>(kScratchFloats) * sizeof(float), M, N, eps, dtype,
                          &cfg, stream);
}
