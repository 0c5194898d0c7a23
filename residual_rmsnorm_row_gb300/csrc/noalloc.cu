// rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot allocate device memory.
//
// The regular backward takes a caller-provided workspace for its per-CTA dw partial sums. Some
// callers have no way to provide one: code that runs while a CUDA graph is being captured (a
// cudaMalloc there fails or breaks the capture), plugins inside an inference engine that owns
// every device allocation, and plain C callers with no caching allocator, for whom a cudaMalloc
// and cudaFree around each call would synchronise the device. This entry point keeps the
// partial sums in a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable of kScratchFloats floats (8 MiB): every GPU that
// loads the library holds it until the process exits. All calls on a device share it, and it
// keeps the previous call's contents; nothing in it needs to start at zero, because stage 1
// writes every element that stage 2 reads. Two calls whose kernels overlap on the GPU (on
// different streams, or from different threads without ordering) race on the array.
//
// Host code cannot use the array's name as a device address, so the first call on each device
// looks the address up with cudaGetSymbolAddress (with that device current) and caches it. That
// lookup is the first call's only extra work; make the first call on a device before any
// stream capture begins.
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
    if (N > kScratchFloats) return RRN_ERR_SCRATCH;  // not even one row of partial sums fits
    if (M == 0 || N < 1) {
        // nothing to launch (or a shape error the regular entry point reports)
        return rmsnorm_bwd(dy, x, w, rstd, dx, dw, nullptr, 0, M, N, eps, dtype, stream);
    }
    // The regular plan, with the number of stage-1 CTAs (one row of partial sums each) lowered
    // until the partial sums fit the array.
    rrn_launch cfg{};
    int st = rrn_plan_bwd(dy, nullptr, x, w, dx, M, N, dtype, &cfg);
    if (st != RRN_OK) return st;
    const int64_t fit = kScratchFloats / N;
    if (cfg.ctas > fit) {
        cfg.ctas = static_cast<int>(fit);
        // a row split over clusters needs whole clusters (it then writes a row per cluster)
        if (cfg.variant == RRN_VARIANT_ROW_CLUSTER) cfg.ctas -= cfg.ctas % cfg.cluster;
    }
    float *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != RRN_OK) return st;
    return rmsnorm_bwd_ex(dy, x, w, rstd, dx, dw, scratch,
                          static_cast<size_t>(kScratchFloats) * sizeof(float), M, N, eps, dtype,
                          &cfg, stream);
}
