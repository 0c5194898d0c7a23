// C ABI of the RMSNorm library: argument validation, launch planning, dispatch.
//
// Every entry point validates all of its arguments before touching the GPU, picks a kernel
// variant from (dtype, M, N, alignment, SM count), launches on the caller's stream and
// returns. Nothing here allocates device memory, synchronises, or compiles code at run time
// (the CuTe DSL skill page's rule for a kernel wrapper - no per-call allocation, copy or
// recompilation, "Workflow 0" step 4 and "Workflow 1" step 5 - applied to a prebuilt
// library).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <map>
#include <mutex>
#include <tuple>

#include "launch.h"
#include "rrn.h"
#include "tma.cuh"

namespace rrn {

// The fault word kernels report a timed-out wait into (one per device, like every __device__
// variable). Kernels get its address as an argument.
__device__ unsigned int g_device_faults = 0;

// One thread waits, with a bound, on an mbarrier that expects an arrival nobody makes.
__global__ void selftest_wait_timeout_kernel(uint64_t limit_ns, unsigned int *faults) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    fence_proxy_async();
    (void)mbar_wait(&bar, 0, faults, limit_ns);
}

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return RRN_ERR_CUDA;
}

// ---------------------------------------------------------------- device properties (cached)
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int current_sm_count(int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < kMaxDevices) {
        int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *sms = cached;
            return RRN_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    *sms = n;
    return RRN_OK;
}

// Device address of the fault word on the current device (looked up once per device).
std::atomic<uintptr_t> g_fault_addr[kMaxDevices];

int fault_word(unsigned int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < kMaxDevices) {
        const uintptr_t a = g_fault_addr[dev].load(std::memory_order_relaxed);
        if (a) {
            *out = reinterpret_cast<unsigned int *>(a);
            return RRN_OK;
        }
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_faults);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < kMaxDevices)
        g_fault_addr[dev].store(reinterpret_cast<uintptr_t>(p), std::memory_order_relaxed);
    *out = static_cast<unsigned int *>(p);
    return RRN_OK;
}

// Occupancy per (device, kernel instance, block size, dynamic shared memory, cluster size),
// computed once.
std::mutex g_occ_mutex;
std::map<std::tuple<int, int, int, int, int, int, int, int, int, int>, int> g_occ;

int occupancy(bool bwd, int dtype, bool fused, const Launch &l) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, bwd ? 1 : 0, dtype, fused ? 1 : 0, l.variant, l.vpt,
                                     l.threads, l.vec ? 1 : 0, l.smem, l.cluster);
    {
        std::lock_guard<std::mutex> g(g_occ_mutex);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = bwd ? (dtype == RRN_BF16 ? occupancy_bwd_bf16(fused, l) : occupancy_bwd_f32(fused, l))
                : (dtype == RRN_BF16 ? occupancy_fwd_bf16(fused, l) : occupancy_fwd_f32(fused, l));
    std::lock_guard<std::mutex> g(g_occ_mutex);
    g_occ[key] = n;
    return n;
}

// Occupancy of a LayerNorm kernel (same cache; the key's `bwd` slot holds 2 + bwd).
int occupancy_ln(bool bwd, int dtype, bool flag, const Launch &l) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, 2 + (bwd ? 1 : 0), dtype, flag ? 1 : 0, l.variant, l.vpt,
                                     l.threads, l.vec ? 1 : 0, l.smem, l.cluster);
    {
        std::lock_guard<std::mutex> g(g_occ_mutex);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    int n = dtype == RRN_BF16 ? occupancy_ln_bf16(bwd, flag, l) : occupancy_ln_f32(bwd, flag, l);
    std::lock_guard<std::mutex> g(g_occ_mutex);
    g_occ[key] = n;
    return n;
}

// ---------------------------------------------------------------- argument checks
int elem_size(int dtype) { return dtype == RRN_BF16 ? 2 : dtype == RRN_F32 ? 4 : 0; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(int64_t M, int64_t N, float eps, int dtype) {
    if (elem_size(dtype) == 0) return RRN_ERR_DTYPE;
    if (M < 0 || N < 1 || N > INT32_MAX) return RRN_ERR_SHAPE;
    if (M > 0 && M > (INT64_MAX / 16) / N) return RRN_ERR_SHAPE;
    if (!std::isfinite(eps) || eps < 0.f) return RRN_ERR_EPS;
    return RRN_OK;
}

int round_up32(int64_t v) { return static_cast<int>((v + 31) / 32 * 32); }

int ceil_pow2_vpt(int64_t need, int max_vpt) {
    int v = 1;
    while (v < need && v < max_vpt) v *= 2;
    return v;
}

int clamp_grid(int64_t v) {
    if (v < 1) return 1;
    return v > INT32_MAX ? INT32_MAX : static_cast<int>(v);
}

// Threads per CTA the row-per-CTA forward aims for on large M (VPT grows with N): measured best
// across N = 4096 and 7168 (narrow CTAs with many vectors per thread, several CTAs per SM).
constexpr int kFwdTargetThreads = 128;
constexpr int kBwdTargetThreads = 256;
// Threads per CTA for few-row (decode) problems: one CTA per row, as wide as this.
constexpr int kDecodeTargetThreads = 512;
// LayerNorm backward of rows split over a cluster: chunks of up to 256 vectors per CTA (clusters
// of 8 from 1024 vectors a row, wider chunks at 8), two vectors a thread. Measured on
// 8192 x 16384 bf16 with the asynchronous exchange and the next row asked into L2: 194 us fused,
// 173 us plain, against 213 / 191 us for clusters of 4 with 2 x 256 and 227 / 208 us with
// 4 x 128. Rows held by one CTA: see ln_bwd_vpt.
constexpr int kLnBwdSplitChunkVec = 256;
constexpr int kLnBwdSplitThreads = 128;
// Narrowest CTA the LayerNorm backward feeds through the TMA ring at 2 vectors per thread;
// narrower ones hold their rows in registers (65536 x 1024 bf16 plain: 96.6 us at 64 threads
// without the ring, 105 with it). At 4 vectors per thread the ring wins at any width
// (32768 x 2048 plain, 64 threads: 92.5 us vs 117).
constexpr int kLnBwdMinRingThreads = 128;
// Widest row (in 128-bit vectors) one CTA holds in registers: 8 vectors x 256 threads.
constexpr int kRowCtaMaxVec = 2048;
// The fused forward takes a row per warp only up to this many vectors: from 129 to 256 vectors
// a row per CTA measured faster (bf16, 64 Mi elements, back to back: 2048 columns 85.7 -> 79.7
// us at 2 x 128, 1536 columns 95.7 -> 87.3 at 2 x 96; the plain forward keeps the row per warp
// up to 256 vectors: 2048 columns 41.8 us against 64.3 for the best row-per-CTA layout).
constexpr int kFwdWarpMaxVecFused = 128;
constexpr int kLnFwdMaxVpt = 4;         // LayerNorm forward row layouts (plan_ln_fwd)
constexpr int kLnFwdTargetThreads = 64;
// fp8 output: one row per warp up to this many vectors over many rows (plan_quant)
constexpr int kQuantWarpMaxVec = 256;
// RMSNorm backward: one row per warp (bwd_row_warp) up to this many vectors over many rows
// (bf16, 64 Mi elements, back to back, against the ring: 512 columns 89.1 -> 71.7 us plain,
// 100.9 -> 88.5 with the gradient at residual_out; 1024 columns 75.1 -> 72.3 plain, while with
// the gradient the ring stays ahead there, 87.6 against 89.2; 2048 columns the ring, 69.3
// against 82.2)
constexpr int kBwdWarpMaxVec = 128;
constexpr int kBwdWarpMaxVecAddGrad = 64;
// LayerNorm backward: one row per warp (ln_bwd_row_warp) up to this many vectors over many rows
// (bf16, back to back, against a row per CTA of 2 vectors a thread: 512 columns 97.2 -> 80.9 us
// plain, 106.9 -> 97.2 with the gradient at residual_out; 1024 columns 91.8 -> 85.0 and
// 101.0 -> 99.0)
constexpr int kLnBwdWarpMaxVec = 128;
// Vectors of a row each CTA of the cluster split takes when the planner chooses the cluster
// size, for the fused forward (two input rows): measured best at 4 vectors x 128 threads a CTA.
// The plain forward (one input row) keeps the same bytes in flight per thread with twice as
// many vectors: measured best at 8 x 128.
constexpr int kClusterChunkVec = 512;

// Vectors per CTA of the forward's row split for a fused or plain forward.
int cluster_chunk_vec(bool fused) { return fused ? kClusterChunkVec : 2 * kClusterChunkVec; }
// Widest row (in vectors) the forward kernels split over a cluster: 8 CTAs of up to 1024 vectors.
// Fused rows of 4096-8192 vectors take chunks above kClusterChunkVec: with the asynchronous
// cluster exchange that measured faster than the two-pass kernel (4096 x 65536 bf16: 365 vs 400
// us; fp32 4096 x 32768: 321 vs 375; fp8 output 294 vs 390).
constexpr int64_t kClusterMaxVec = static_cast<int64_t>(kMaxCluster) * 2 * kClusterChunkVec;
// CTAs per cluster for the backward's distributed-shared-memory pre-reduction of dw when the
// caller leaves the choice to the planner (0: no clusters).
constexpr int kBwdCluster = 0;

// Largest dynamic shared memory one CTA may use (sm_100-class parts: 227 KB).
constexpr int kMaxDynSmem = 227 * 1024;

// Pick the ring depth for a TMA variant whose one-row slot takes `slot_bytes`. Resident CTAs
// per SM come first (measured on the 16384 x 4096 bf16 backward: 4 CTAs x 2 stages 71.8 us,
// 2 CTAs x 7 stages 96.8 us), at most `max_occ` of them when that is positive; among the
// depths that keep the most CTAs resident, the shallowest from 2 up that keeps kRingTargetBytes
// of ring per SM - `capped_target` when max_occ held the CTAs back - (else the deepest of
// them). Returns the CTAs per SM (0: no depth fits); sets l->stages and l->smem.
constexpr int64_t kRingTargetBytes = 64 * 1024;

// The backward with two input rows (x, dy) measured best with at most about 48 KB of rows being
// worked on per SM (resident CTAs x slot bytes, at least 2 CTAs) and, where that holds CTAs
// back, a ring of about 128 KB per SM to keep the bytes in flight (bf16, 64 Mi elements per
// matrix, back to back): 3072 columns 73.3 -> 69.2 us (4 CTAs x 3 stages instead of 5 x 2),
// 4096 columns 73.5 -> 68.0 (3 x 3 instead of 4 x 2), 6144 columns 71.5 -> 69.5 (2 x 3 instead
// of 2 x 2); 1024, 2048 and 8192 columns kept their layouts (there 3 or 4 stages measured 1-2 %
// slower). With a third input row the most CTAs and 64 KB of ring per SM stayed the best
// measured at every width.
constexpr int64_t kBwdPlainWorkBytes = 48 * 1024;
constexpr int64_t kBwdPlainRingBytes = 128 * 1024;

// occ(t): resident CTAs per SM of launch t.
template <typename Occ>
int plan_ring(Occ occ, int slot_bytes, int want_stages, Launch *l, int max_occ = 0,
              int64_t capped_target = kRingTargetBytes) {
    int occ_of[kMaxStages + 1] = {};
    int best_occ = 0;
    bool capped = false;
    for (int S = 1; S <= kMaxStages; ++S) {
        if (want_stages && S != want_stages) continue;
        const int64_t smem = static_cast<int64_t>(S) * slot_bytes;
        if (smem > kMaxDynSmem) break;
        Launch t = *l;
        t.stages = S;
        t.smem = static_cast<int>(smem);
        occ_of[S] = occ(t);
        if (max_occ > 0 && occ_of[S] >= max_occ) {
            occ_of[S] = max_occ;
            capped = true;
        }
        if (occ_of[S] > best_occ) best_occ = occ_of[S];
    }
    if (best_occ < 1) return 0;
    const int64_t target = capped && best_occ == max_occ ? capped_target : kRingTargetBytes;
    int pick = 0;
    for (int S = 1; S <= kMaxStages; ++S) {
        if (occ_of[S] != best_occ) continue;
        pick = S;
        if (S >= 2 && static_cast<int64_t>(best_occ) * S * slot_bytes >= target) break;
    }
    l->stages = pick;
    l->smem = pick * slot_bytes;
    return best_occ;
}

// The layout of a row-per-warp kernel (every op's ROW_WARP variant): a lane takes vpt vectors
// (given, or the smallest power of two covering the row with 32 lanes), 128 threads a CTA unless
// given (at most 256, a multiple of 32). The grid is the caller's: one row per warp for the
// forwards, resident CTAs for the backwards.
int warp_row_layout(int64_t nvec, const rrn_launch *cfg, Launch *l) {
    l->vpt = cfg && cfg->vpt ? cfg->vpt : ceil_pow2_vpt((nvec + 31) / 32, kMaxVpt);
    if (l->vpt != 1 && l->vpt != 2 && l->vpt != 4 && l->vpt != 8) return RRN_ERR_CONFIG;
    if (static_cast<int64_t>(l->vpt) * 32 < nvec) return RRN_ERR_CONFIG;
    l->threads = cfg && cfg->threads ? cfg->threads : 128;
    if (l->threads < 32 || l->threads % 32 || l->threads > 256) return RRN_ERR_CONFIG;
    return RRN_OK;
}

// ---------------------------------------------------------------- forward planning
// True when every row of every matrix starts on a 16-byte boundary (128-bit vector path).
bool vec_path_ok(std::initializer_list<const void *> ptrs, int64_t N, int dtype) {
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return false;
    return N % (16 / elem_size(dtype)) == 0;
}

// The layout of a forward-type kernel with each row split over a cluster (fwd_row_cluster,
// quant_row_cluster): the cluster size from cluster_chunk_vec unless given (8 for wider rows), the
// vectors per thread as the row-per-CTA forward picks them for one CTA's chunk with about
// `target_threads` threads, and - unless given - one wave of clusters: as many as the GPU holds
// at once (`occ` gives that number for a layout).
template <typename Occ>
int fwd_cluster_layout(int64_t nvec, int64_t M, bool fused, const rrn_launch *cfg, Occ occ, Launch *l,
                       int target_threads = kFwdTargetThreads) {
    if (cfg && cfg->cluster) {
        l->cluster = cfg->cluster;
    } else {
        l->cluster = 2;
        while (l->cluster < kMaxCluster && nvec > static_cast<int64_t>(l->cluster) * cluster_chunk_vec(fused)) l->cluster *= 2;
    }
    if (l->cluster < 2 || l->cluster > kMaxCluster) return RRN_ERR_CONFIG;
    const int64_t chunk = (nvec + l->cluster - 1) / l->cluster;
    if (cfg && cfg->vpt) {
        l->vpt = cfg->vpt;
    } else {
        l->vpt = ceil_pow2_vpt((chunk + target_threads - 1) / target_threads, kMaxVpt);
        while (l->vpt < kMaxVpt && chunk > static_cast<int64_t>(l->vpt) * fwd_max_threads(l->vpt)) l->vpt *= 2;
    }
    l->threads = cfg && cfg->threads ? cfg->threads : round_up32((chunk + l->vpt - 1) / l->vpt);
    if (l->vpt != 1 && l->vpt != 2 && l->vpt != 4 && l->vpt != 8) return RRN_ERR_CONFIG;
    if (l->threads < 32 || l->threads % 32 || l->threads > fwd_max_threads(l->vpt)) return RRN_ERR_CONFIG;
    if (static_cast<int64_t>(l->vpt) * l->threads < chunk) return RRN_ERR_CONFIG;
    if (cfg && cfg->ctas) {
        l->ctas = cfg->ctas;
        if (l->ctas % l->cluster) return RRN_ERR_CONFIG;
    } else {
        int64_t clusters = occ(*l);
        if (clusters < 1) clusters = 1;
        if (clusters > M) clusters = M;
        if (clusters > INT32_MAX / l->cluster) clusters = INT32_MAX / l->cluster;
        l->ctas = static_cast<int>(clusters) * l->cluster;
    }
    return RRN_OK;
}

int plan_fwd_impl(bool vec_ok, bool fused, int64_t M, int64_t N, int dtype, const rrn_launch *cfg,
                  Launch *out) {
    const int V = 16 / elem_size(dtype);
    const int64_t nvec = N / V;
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != RRN_OK) return st;

    Launch l{};
    l.variant = cfg && cfg->variant ? cfg->variant : RRN_VARIANT_AUTO;
    if (l.variant == RRN_VARIANT_AUTO) {
        // Measured on bf16 rows of 4096 to 262144 columns, fused and plain: one row per CTA
        // while the CTA holds the row - fused up to 1024 vectors (8 a thread x 128 threads),
        // plain up to kRowCtaMaxVec (8 x 256: the same bytes in flight per thread); wider rows
        // split over a cluster, cluster_chunk_vec vectors per CTA; wider still, the two-pass
        // kernel. Few rows (decode): one CTA per row up to kRowCtaMaxVec.
        const bool few = M < 2LL * sms;
        const int64_t cta_max = few || !fused ? kRowCtaMaxVec : 128 * kMaxVpt;
        if (!vec_ok) l.variant = RRN_VARIANT_STREAM;
        else if (nvec <= (fused ? kFwdWarpMaxVecFused : 32 * kMaxVpt) && M >= 4LL * sms) l.variant = RRN_VARIANT_ROW_WARP;
        else if (nvec <= cta_max) l.variant = RRN_VARIANT_ROW_CTA;
        else if (nvec <= kClusterMaxVec) l.variant = RRN_VARIANT_ROW_CLUSTER;
        else l.variant = RRN_VARIANT_STREAM;
    }
    l.vec = (l.variant == RRN_VARIANT_STREAM) ? vec_ok : true;
    l.stages = 0;
    l.smem = 0;
    l.cluster = 0;

    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA: {
            if (!vec_ok) return RRN_ERR_CONFIG;
            if (cfg && cfg->vpt) {
                l.vpt = cfg->vpt;
            } else if (M < 2LL * sms) {
                // Few rows (decode shapes): one wide CTA per row, each row arriving in one round
                // trip; 512 threads measured faster than 1024 (M = 1..64 x 8192, bf16 and fp32).
                l.vpt = ceil_pow2_vpt((nvec + kDecodeTargetThreads - 1) / kDecodeTargetThreads, kMaxVpt);
                while (l.vpt < kMaxVpt && nvec > static_cast<int64_t>(l.vpt) * fwd_max_threads(l.vpt)) l.vpt *= 2;
            } else {
                l.vpt = ceil_pow2_vpt((nvec + kFwdTargetThreads - 1) / kFwdTargetThreads, kMaxVpt);
                while (l.vpt < kMaxVpt && nvec > static_cast<int64_t>(l.vpt) * fwd_max_threads(l.vpt)) l.vpt *= 2;
            }
            l.threads = cfg && cfg->threads ? cfg->threads : round_up32((nvec + l.vpt - 1) / l.vpt);
            if (l.vpt != 1 && l.vpt != 2 && l.vpt != 4 && l.vpt != 8) return RRN_ERR_CONFIG;
            if (l.threads < 32 || l.threads % 32 || l.threads > fwd_max_threads(l.vpt)) return RRN_ERR_CONFIG;
            if (static_cast<int64_t>(l.vpt) * l.threads < nvec) return RRN_ERR_CONFIG;
            l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid(M);
            break;
        }
        case RRN_VARIANT_ROW_WARP: {
            if (!vec_ok) return RRN_ERR_CONFIG;
            st = warp_row_layout(nvec, cfg, &l);
            if (st != RRN_OK) return st;
            l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid((M + l.threads / 32 - 1) / (l.threads / 32));
            break;
        }
        case RRN_VARIANT_ROW_CLUSTER: {
            if (!vec_ok) return RRN_ERR_CONFIG;
            st = fwd_cluster_layout(nvec, M, fused, cfg, [&](const Launch &t) { return occupancy(false, dtype, fused, t); },
                                    &l);
            if (st != RRN_OK) return st;
            break;
        }
        case RRN_VARIANT_ROW_TMA: {
            if (!vec_ok) return RRN_ERR_CONFIG;
            if (cfg && cfg->vpt) {
                l.vpt = cfg->vpt;
            } else {
                l.vpt = ceil_pow2_vpt((nvec + kFwdTargetThreads - 1) / kFwdTargetThreads, kMaxVpt);
                while (l.vpt < kMaxVpt && nvec > static_cast<int64_t>(l.vpt) * fwd_max_threads(l.vpt)) l.vpt *= 2;
            }
            l.threads = cfg && cfg->threads ? cfg->threads : round_up32((nvec + l.vpt - 1) / l.vpt);
            if (l.vpt != 1 && l.vpt != 2 && l.vpt != 4 && l.vpt != 8) return RRN_ERR_CONFIG;
            if (l.threads < 32 || l.threads % 32 || l.threads > fwd_max_threads(l.vpt)) return RRN_ERR_CONFIG;
            if (static_cast<int64_t>(l.vpt) * l.threads < nvec) return RRN_ERR_CONFIG;
            const int want = cfg ? cfg->stages : 0;
            if (want < 0 || want > kMaxStages) return RRN_ERR_CONFIG;
            const int64_t slot = (fused ? 2 : 1) * N * elem_size(dtype);
            if (slot > kMaxDynSmem) return RRN_ERR_CONFIG;
            const int occ = plan_ring([&](const Launch &t) { return occupancy(false, dtype, fused, t); },
                                      static_cast<int>(slot), want, &l);
            if (occ < 1) return RRN_ERR_CONFIG;
            l.ctas = cfg && cfg->ctas ? cfg->ctas
                                      : clamp_grid(M < static_cast<int64_t>(sms) * occ ? M : static_cast<int64_t>(sms) * occ);
            break;
        }
        case RRN_VARIANT_STREAM: {
            l.vpt = 1;
            const int64_t chunks = l.vec ? nvec : N;
            // 1024 threads measured faster from 8192 chunks a row (4096 x 65536, 1024 x 262144)
            l.threads = cfg && cfg->threads ? cfg->threads
                                            : (chunks >= 8192 ? 1024 : chunks >= 512 ? 512 : round_up32(chunks));
            if (l.threads < 32 || l.threads % 32 || l.threads > 1024) return RRN_ERR_CONFIG;
            if (cfg && cfg->ctas) {
                l.ctas = cfg->ctas;
            } else {
                const int occ = occupancy(false, dtype, fused, l);
                l.ctas = clamp_grid(M < static_cast<int64_t>(sms) * (occ > 0 ? occ : 1)
                                        ? M
                                        : static_cast<int64_t>(sms) * (occ > 0 ? occ : 1));
            }
            break;
        }
        default:
            return RRN_ERR_CONFIG;
    }
    if (l.ctas < 1) return RRN_ERR_CONFIG;
    *out = l;
    return RRN_OK;
}

int check_fwd(const void *x, const void *res, const void *res_out, const void *w, const void *y,
              const float *rstd, int64_t M, int64_t N, float eps, int dtype) {
    int st = check_common(M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return RRN_OK;  // nothing is read or written: pointers are not examined
    if (!x || !w || !y || (res && !res_out)) return RRN_ERR_NULL;
    const uintptr_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(w, es) || !aligned(y, es) || (res && !aligned(res, es)) ||
        (res && !aligned(res_out, es)) || (rstd && !aligned(rstd, 4)))
        return RRN_ERR_ALIGN;
    return RRN_OK;
}

int run_fwd(const void *x, const void *res, void *res_out, const void *w, void *y, float *rstd,
            int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg, cudaStream_t stream) {
    int st = check_fwd(x, res, res_out, w, y, rstd, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return RRN_OK;
    Launch l;
    st = plan_fwd_impl(vec_path_ok({x, res, res_out, w, y}, N, dtype), res != nullptr, M, N, dtype,
                       cfg, &l);
    if (st != RRN_OK) return st;
    unsigned int *faults = nullptr;
    st = fault_word(&faults);
    if (st != RRN_OK) return st;
    FwdArgs a{x, res, res ? res_out : nullptr, w, y, rstd, M, static_cast<int>(N), eps, 0, faults};
    cudaError_t e = dtype == RRN_BF16 ? launch_fwd_bf16(a, l, stream) : launch_fwd_f32(a, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

// ---------------------------------------------------------------- backward planning
// add_grad: the fused backward (a third input row, the gradient at residual_out).
// Rows of partial sums the RMSNorm backward's stage 1 writes (and its workspace must hold): one
// per CTA, or one per cluster when the CTAs work in clusters.
int bwd_partial_rows(const Launch &l) { return l.cluster ? l.ctas / l.cluster : l.ctas; }

int plan_bwd_impl(bool vec_ok, bool add_grad, int64_t M, int64_t N, int dtype,
                  const rrn_launch *cfg, Launch *out, int64_t *rows_per_cta) {
    const int V = 16 / elem_size(dtype);
    const int64_t nvec = N / V;
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != RRN_OK) return st;

    Launch l{};
    l.variant = cfg && cfg->variant ? cfg->variant : RRN_VARIANT_AUTO;
    if (l.variant == RRN_VARIANT_AUTO) {
        const bool regs = vec_ok && nvec <= static_cast<int64_t>(kBwdMaxVpt) * bwd_max_threads(kBwdMaxVpt);
        // The TMA ring (rows and the next rstd requested ahead) measured faster than the
        // register variant for two and three input rows; rows whose ring slot would take more
        // than half the shared memory use the register variant.
        // Rows too wide for that: split over a thread-block cluster up to kMaxCluster chunks of
        // kClusterChunkVec vectors (4 a thread x 128 threads, as the ring's CTAs), else the
        // two-pass kernel.
        const int64_t slot = (add_grad ? 3 : 2) * N * elem_size(dtype);
        const int64_t warp_max = add_grad ? kBwdWarpMaxVecAddGrad : kBwdWarpMaxVec;
        l.variant = regs ? (nvec <= warp_max && M >= 4LL * sms ? RRN_VARIANT_ROW_WARP
                            : slot <= kMaxDynSmem / 2                ? RRN_VARIANT_ROW_TMA
                                                                     : RRN_VARIANT_ROW_CTA)
                  : vec_ok && nvec <= static_cast<int64_t>(kMaxCluster) * kClusterChunkVec ? RRN_VARIANT_ROW_CLUSTER
                                                                                           : RRN_VARIANT_STREAM;
    }
    l.vec = (l.variant == RRN_VARIANT_STREAM) ? vec_ok : true;
    l.stages = 0;
    l.smem = 0;
    l.cluster = 0;
    int ring_occ = 0;
    switch (l.variant) {
        case RRN_VARIANT_ROW_CLUSTER: {
            // Each row split across l.cluster CTAs; the grid is the clusters resident at once
            // (at most M), cluster k walking rows k, k + K, ...; the workspace gets K rows.
            if (!vec_ok) return RRN_ERR_CONFIG;
            if (cfg && cfg->cluster) {
                l.cluster = cfg->cluster;
            } else {
                l.cluster = 2;
                while (l.cluster < kMaxCluster && nvec > static_cast<int64_t>(l.cluster) * kClusterChunkVec) l.cluster *= 2;
            }
            if (l.cluster < 2 || l.cluster > kMaxCluster) return RRN_ERR_CONFIG;
            const int64_t chunk = (nvec + l.cluster - 1) / l.cluster;
            if (cfg && cfg->vpt) {
                l.vpt = cfg->vpt;
            } else {
                l.vpt = ceil_pow2_vpt((chunk + 127) / 128, kBwdMaxVpt);
                while (l.vpt < kBwdMaxVpt && chunk > static_cast<int64_t>(l.vpt) * bwd_max_threads(l.vpt)) l.vpt *= 2;
            }
            if (l.vpt != 1 && l.vpt != 2 && l.vpt != 4) return RRN_ERR_CONFIG;
            l.threads = cfg && cfg->threads ? cfg->threads : round_up32((chunk + l.vpt - 1) / l.vpt);
            if (l.threads < 32 || l.threads % 32 || l.threads > bwd_max_threads(l.vpt)) return RRN_ERR_CONFIG;
            if (static_cast<int64_t>(l.vpt) * l.threads < chunk) return RRN_ERR_CONFIG;
            if (cfg && cfg->ctas) {
                l.ctas = cfg->ctas;
                if (l.ctas % l.cluster) return RRN_ERR_CONFIG;
            } else {
                int64_t clusters = occupancy(true, dtype, add_grad, l);
                if (clusters < 1) clusters = 1;
                if (clusters > M) clusters = M;
                if (clusters > INT32_MAX / l.cluster) clusters = INT32_MAX / l.cluster;
                l.ctas = M == 0 ? 0 : static_cast<int>(clusters) * l.cluster;
            }
            *rows_per_cta = M == 0 ? 0 : (M + l.ctas / l.cluster - 1) / (l.ctas / l.cluster);
            *out = l;
            return RRN_OK;
        }
        case RRN_VARIANT_ROW_TMA:
        case RRN_VARIANT_ROW_CTA: {
            if (!vec_ok) return RRN_ERR_CONFIG;
            if (cfg && cfg->vpt) {
                l.vpt = cfg->vpt;
            } else {
                // the TMA ring measured best with narrower CTAs (more of them per SM)
                const int target = l.variant == RRN_VARIANT_ROW_TMA ? 128 : kBwdTargetThreads;
                l.vpt = ceil_pow2_vpt((nvec + target - 1) / target, kBwdMaxVpt);
                while (l.vpt < kBwdMaxVpt && nvec > static_cast<int64_t>(l.vpt) * bwd_max_threads(l.vpt)) l.vpt *= 2;
            }
            if (l.vpt != 1 && l.vpt != 2 && l.vpt != 4) return RRN_ERR_CONFIG;
            l.threads = cfg && cfg->threads ? cfg->threads : round_up32((nvec + l.vpt - 1) / l.vpt);
            if (l.threads < 32 || l.threads % 32 || l.threads > bwd_max_threads(l.vpt)) return RRN_ERR_CONFIG;
            if (static_cast<int64_t>(l.vpt) * l.threads < nvec) return RRN_ERR_CONFIG;
            if (l.variant == RRN_VARIANT_ROW_TMA) {
                const int want = cfg ? cfg->stages : 0;
                if (want < 0 || want > kMaxStages) return RRN_ERR_CONFIG;
                const int64_t slot = (add_grad ? 3 : 2) * N * elem_size(dtype);
                if (slot > kMaxDynSmem) return RRN_ERR_CONFIG;
                const int64_t work_cap = kBwdPlainWorkBytes / slot;
                ring_occ = plan_ring([&](const Launch &t) { return occupancy(true, dtype, add_grad, t); },
                                     static_cast<int>(slot), want, &l,
                                     add_grad ? 0 : static_cast<int>(work_cap < 2 ? 2 : work_cap),
                                     kBwdPlainRingBytes);
                if (ring_occ < 1) return RRN_ERR_CONFIG;
            }
            break;
        }
        case RRN_VARIANT_ROW_WARP: {
            // a row per warp; the CTA's warps add their dw sums in N floats of shared memory
            if (!vec_ok) return RRN_ERR_CONFIG;
            st = warp_row_layout(nvec, cfg, &l);
            if (st != RRN_OK) return st;
            l.smem = static_cast<int>(N * static_cast<int64_t>(sizeof(float)));
            break;
        }
        case RRN_VARIANT_STREAM: {
            l.vpt = 1;
            const int64_t chunks = l.vec ? nvec : N;
            l.threads = cfg && cfg->threads ? cfg->threads
                                            : (chunks >= 512 ? 512 : round_up32(chunks));
            if (l.threads < 32 || l.threads % 32 || l.threads > 1024) return RRN_ERR_CONFIG;
            break;
        }
        default:
            return RRN_ERR_CONFIG;
    }
    int64_t want = 0;
    if (cfg && cfg->ctas) {
        want = cfg->ctas;
    } else {
        const int occ = ring_occ ? ring_occ : occupancy(true, dtype, add_grad, l);
        want = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
    }
    if (want < 1) return RRN_ERR_CONFIG;
    // Register and TMA stage 1 may pre-reduce the dw partial sums over clusters of C CTAs
    // (distributed shared memory), so that stage 2 reads P / C rows. cfg->cluster: 0 = the
    // planner's choice (kBwdCluster), 1 = no clusters, 2, 4 or 8 = that size.
    int C = cfg && cfg->cluster ? cfg->cluster : kBwdCluster;
    if (C != 0 && C != 1 && C != 2 && C != 4 && C != 8) return RRN_ERR_CONFIG;
    if (C == 1 || (l.variant != RRN_VARIANT_ROW_CTA && l.variant != RRN_VARIANT_ROW_TMA)) C = 0;
    Launch lc = l;
    if (C) {
        lc.cluster = C;
        if (l.variant == RRN_VARIANT_ROW_CTA) lc.smem = static_cast<int>(N * sizeof(float));
        if (!(cfg && cfg->ctas)) {
            // clusters are placed within one GPC: keep P to one wave of them
            const int clusters = occupancy(true, dtype, add_grad, lc);
            if (clusters < 1) return RRN_ERR_CONFIG;
            if (want > static_cast<int64_t>(clusters) * C) want = static_cast<int64_t>(clusters) * C;
        }
    }
    // CTA p takes rows p, p + P, ...: with P <= M every CTA owns at least one row (so every
    // workspace row stage 2 reads is written).
    l.ctas = M == 0 ? 0 : clamp_grid(want < M ? want : M);
    if (C && l.ctas >= 2 * C) {
        lc.ctas = l.ctas / C * C;  // P a multiple of the cluster size
        l = lc;
    }
    *rows_per_cta = M == 0 ? 0 : (M + l.ctas - 1) / l.ctas;
    *out = l;
    return RRN_OK;
}

int check_bwd(const void *dy, const void *d_ro, const void *x, const void *w, const float *rstd,
              const void *dx, const float *dw, int64_t M, int64_t N, float eps, int dtype) {
    int st = check_common(M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return RRN_OK;  // no row is read or written: row pointers are not examined
    if (!dy || !x || !w || !rstd || !dx || !dw) return RRN_ERR_NULL;
    const uintptr_t es = elem_size(dtype);
    if (!aligned(dy, es) || !aligned(x, es) || !aligned(w, es) || !aligned(dx, es) ||
        (d_ro && !aligned(d_ro, es)) || !aligned(rstd, 4) || !aligned(dw, 4))
        return RRN_ERR_ALIGN;
    return RRN_OK;
}

// M == 0: dw (and db) are sums over no rows, so they are set to zero on the stream; no row
// data is examined.
int zero_sums(float *dw, float *db, int64_t N, cudaStream_t stream) {
    if (!dw) return RRN_ERR_NULL;
    if (!aligned(dw, 4) || (db && !aligned(db, 4))) return RRN_ERR_ALIGN;
    for (float *p : {dw, db}) {
        if (!p) continue;
        const cudaError_t e = cudaMemsetAsync(p, 0, static_cast<size_t>(N) * sizeof(float), stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return RRN_OK;
}

int run_bwd(const void *dy, const void *d_ro, const void *x, const void *w, const float *rstd,
            void *dx, float *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
            float eps, int dtype, const rrn_launch *cfg, cudaStream_t stream) {
    int st = check_bwd(dy, d_ro, x, w, rstd, dx, dw, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return zero_sums(dw, nullptr, N, stream);
    Launch l;
    int64_t rpc = 0;
    st = plan_bwd_impl(vec_path_ok({dy, d_ro, x, w, dx}, N, dtype), d_ro != nullptr, M, N, dtype,
                       cfg, &l, &rpc);
    if (st != RRN_OK) return st;
    const size_t need = static_cast<size_t>(bwd_partial_rows(l)) * static_cast<size_t>(N) * sizeof(float);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return RRN_ERR_WORKSPACE;
    unsigned int *faults = nullptr;
    st = fault_word(&faults);
    if (st != RRN_OK) return st;
    BwdArgs a{dy, d_ro, x, w, rstd, dx, dw, static_cast<float *>(workspace), M,
              static_cast<int>(N), 0, faults};
    cudaError_t e = dtype == RRN_BF16 ? launch_bwd_bf16(a, l, stream) : launch_bwd_f32(a, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

// ---------------------------------------------------------------- LayerNorm
// Register layout (vpt, threads) for a row of nvec vectors, as the RMSNorm planners choose it:
// about kDecodeTargetThreads threads for few rows, about target_threads otherwise.
int pick_row_layout(int64_t nvec, int64_t M, int sms, const rrn_launch *cfg, int max_vpt,
                    int (*max_threads)(int), int target_threads, Launch *l) {
    if (cfg && cfg->vpt) {
        l->vpt = cfg->vpt;
    } else {
        const int target = M < 2LL * sms ? kDecodeTargetThreads : target_threads;
        l->vpt = ceil_pow2_vpt((nvec + target - 1) / target, max_vpt);
        while (l->vpt < max_vpt && nvec > static_cast<int64_t>(l->vpt) * max_threads(l->vpt)) l->vpt *= 2;
    }
    if (l->vpt < 1 || l->vpt > max_vpt || (l->vpt & (l->vpt - 1))) return RRN_ERR_CONFIG;
    l->threads = cfg && cfg->threads ? cfg->threads : round_up32((nvec + l->vpt - 1) / l->vpt);
    if (l->threads < 32 || l->threads % 32 || l->threads > max_threads(l->vpt)) return RRN_ERR_CONFIG;
    if (static_cast<int64_t>(l->vpt) * l->threads < nvec) return RRN_ERR_CONFIG;
    return RRN_OK;
}

int fwd_threads_limit(int vpt) { return fwd_max_threads(vpt); }
int bwd_threads_limit(int vpt) { return bwd_max_threads(vpt); }

int plan_ln_fwd(bool vec_ok, bool fused, int64_t M, int64_t N, int dtype, const rrn_launch *cfg,
                Launch *out) {
    const int64_t nvec = N / (16 / elem_size(dtype));
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != RRN_OK) return st;
    Launch l{};
    l.variant = cfg && cfg->variant ? cfg->variant : RRN_VARIANT_AUTO;
    if (l.variant == RRN_VARIANT_AUTO) {
        // Measured on bf16 rows with a residual and bias (64 Mi elements, back to back): a row
        // per warp up to 128 vectors over many rows (512 columns 200.9 -> 84.6 us, 768 142.9 ->
        // 95.1, 1024 120.6 -> 85.7 against a row per CTA; 2048: 96.2 against 86.6 for a CTA of
        // 4 x 64), a row per CTA up to kRowCtaMaxVec, the two-pass kernel beyond.
        if (!vec_ok) l.variant = RRN_VARIANT_STREAM;
        else if (nvec <= 32 * kLnFwdMaxVpt && M >= 4LL * sms) l.variant = RRN_VARIANT_ROW_WARP;
        else if (nvec <= kRowCtaMaxVec) l.variant = RRN_VARIANT_ROW_CTA;
        else l.variant = RRN_VARIANT_STREAM;
    }
    l.vec = l.variant == RRN_VARIANT_STREAM ? vec_ok : true;
    if (l.variant == RRN_VARIANT_ROW_CTA) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        // 4 vectors a thread (more threads instead) from 256 vectors up: the LayerNorm row
        // kernel keeps more per-row state than RMSNorm's, and 8 vectors a thread took 141-175
        // registers, 2 CTAs per SM (bf16 with a residual and bias, back to back: 6144 columns
        // 135.4 -> 84.8 us at 4 x 192, 8192 columns 109.7 -> 85.3 at 4 x 256, 12288 columns
        // 149.1 -> 88.5 at 4 x 384; 2048 columns 92.9 -> 86.6 at 4 x 64 instead of 2 x 128)
        // (given explicitly, 8 vectors a thread still run)
        st = pick_row_layout(nvec, M, sms, cfg, cfg && cfg->vpt ? kMaxVpt : kLnFwdMaxVpt, fwd_threads_limit,
                             kLnFwdTargetThreads, &l);
        if (st != RRN_OK) return st;
        l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid(M);
    } else if (l.variant == RRN_VARIANT_ROW_WARP) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        st = warp_row_layout(nvec, cfg, &l);
        if (st != RRN_OK) return st;
        l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid((M + l.threads / 32 - 1) / (l.threads / 32));
    } else if (l.variant == RRN_VARIANT_STREAM) {
        l.vpt = 1;
        const int64_t chunks = l.vec ? nvec : N;
        l.threads = cfg && cfg->threads ? cfg->threads : (chunks >= 512 ? 512 : round_up32(chunks));
        if (l.threads < 32 || l.threads % 32 || l.threads > 1024) return RRN_ERR_CONFIG;
        if (cfg && cfg->ctas) {
            l.ctas = cfg->ctas;
        } else {
            const int occ = occupancy_ln(false, dtype, fused, l);
            const int64_t cap = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
            l.ctas = clamp_grid(M < cap ? M : cap);
        }
    } else {
        return RRN_ERR_CONFIG;  // the LayerNorm forward runs the row-per-CTA, row-per-warp and two-pass variants
    }
    if (l.ctas < 1) return RRN_ERR_CONFIG;
    *out = l;
    return RRN_OK;
}

// Vectors per thread of the LayerNorm backward with whole rows in one CTA, chosen by
// measurement over 1024-8192 bf16 columns (128 MB per input matrix; ln_bwd_row_tma reading rows
// twice from its ring): with the gradient at residual_out (a third input row) 2 up to 512
// vectors a row and 4 above (8192 columns: 113 us vs 127 at 2), without it 2 below 256 vectors
// and 4 from there (2048 columns: 92.5 us vs 98.8 at 2) - within 2 % of the best layout measured
// at every width.
int ln_bwd_vpt(int64_t nvec, bool add_grad) {
    int vpt = (add_grad ? nvec <= 512 : nvec < 256) ? 2 : 4;
    while (vpt < kBwdMaxVpt && nvec > static_cast<int64_t>(vpt) * bwd_max_threads(vpt)) vpt *= 2;
    return vpt;
}

int plan_ln_bwd(bool vec_ok, bool add_grad, int64_t M, int64_t N, int dtype, const rrn_launch *cfg,
                Launch *out, int64_t *rows_per_cta) {
    const int64_t nvec = N / (16 / elem_size(dtype));
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != RRN_OK) return st;
    Launch l{};
    l.variant = cfg && cfg->variant ? cfg->variant : RRN_VARIANT_AUTO;
    const int64_t slot = (add_grad ? 3 : 2) * N * elem_size(dtype);
    if (l.variant == RRN_VARIANT_AUTO) {
        // wider rows than one CTA's dw and db registers hold: split over a cluster, as the
        // RMSNorm backward (measured 0.9 TB/s for the two-pass kernel on 8192 x 16384)
        const bool regs = vec_ok && nvec <= static_cast<int64_t>(kBwdMaxVpt) * bwd_max_threads(kBwdMaxVpt);
        const int vpt = ln_bwd_vpt(nvec, add_grad);
        const bool ring = slot <= kMaxDynSmem / 2 &&
                          (vpt >= 4 || round_up32((nvec + vpt - 1) / vpt) >= kLnBwdMinRingThreads);
        l.variant = regs ? (nvec <= kLnBwdWarpMaxVec && M >= 4LL * sms ? RRN_VARIANT_ROW_WARP
                            : ring                                     ? RRN_VARIANT_ROW_TMA
                                                                       : RRN_VARIANT_ROW_CTA)
                  : vec_ok && nvec <= static_cast<int64_t>(kMaxCluster) * kClusterChunkVec ? RRN_VARIANT_ROW_CLUSTER
                                                                                           : RRN_VARIANT_STREAM;
    }
    l.vec = l.variant == RRN_VARIANT_STREAM ? vec_ok : true;
    int ring_occ = 0;
    if (l.variant == RRN_VARIANT_ROW_CLUSTER) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        if (cfg && cfg->cluster) {
            l.cluster = cfg->cluster;
        } else {
            l.cluster = 2;
            while (l.cluster < kMaxCluster && nvec > static_cast<int64_t>(l.cluster) * kLnBwdSplitChunkVec) l.cluster *= 2;
        }
        if (l.cluster < 2 || l.cluster > kMaxCluster) return RRN_ERR_CONFIG;
        const int64_t chunk = (nvec + l.cluster - 1) / l.cluster;
        // two vectors a thread while a CTA of up to 512 threads covers the chunk (4096 x 32768:
        // 220 us fused, 202 plain at 2 x 256 against 246 / 228 at 4 x 128)
        rrn_launch pick = cfg ? *cfg : rrn_launch{};
        if (!pick.vpt && !pick.threads) pick.vpt = chunk <= 2 * bwd_max_threads(2) ? 2 : kBwdMaxVpt;
        st = pick_row_layout(chunk, 1LL << 40, sms, &pick, kBwdMaxVpt, bwd_threads_limit, kLnBwdSplitThreads, &l);
        if (st != RRN_OK) return st;
        if (cfg && cfg->ctas) {
            l.ctas = cfg->ctas;
            if (l.ctas % l.cluster) return RRN_ERR_CONFIG;
        } else {
            int64_t clusters = occupancy_ln(true, dtype, add_grad, l);
            if (clusters < 1) clusters = 1;
            if (clusters > M) clusters = M;
            if (clusters > INT32_MAX / l.cluster) clusters = INT32_MAX / l.cluster;
            l.ctas = M == 0 ? 0 : static_cast<int>(clusters) * l.cluster;
        }
        *rows_per_cta = M == 0 ? 0 : (M + l.ctas / l.cluster - 1) / (l.ctas / l.cluster);
        *out = l;
        return RRN_OK;
    }
    if (l.variant == RRN_VARIANT_ROW_CTA || l.variant == RRN_VARIANT_ROW_TMA) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        rrn_launch pick = cfg ? *cfg : rrn_launch{};
        if (!pick.vpt && !pick.threads) pick.vpt = ln_bwd_vpt(nvec, add_grad);
        // (given only the threads, the vectors per thread are fitted to them)
        st = pick_row_layout(nvec, 1LL << 40, sms, &pick, kBwdMaxVpt, bwd_threads_limit,
                             pick.threads ? pick.threads : bwd_max_threads(1), &l);
        if (st != RRN_OK) return st;
        if (l.variant == RRN_VARIANT_ROW_TMA) {
            // The ring refills a slot one row late (ln_bwd_row_tma), so it needs 2 stages or
            // more: S - 1 rows in flight. Measured back to back with as many CTAs per SM as fit,
            // bf16: 2 stages with or without the gradient at residual_out (16384 x 4096: 92.5 us
            // fused vs 95.1 at 3, 77.2 plain vs 84.9; 32768 x 2048 fused: 92.0 vs 94.5).
            const int want = cfg ? cfg->stages : 0;
            if (want < 0 || want == 1 || want > kMaxStages || 2 * slot > kMaxDynSmem) return RRN_ERR_CONFIG;
            const int S = want ? want : 2;
            if (S * slot > kMaxDynSmem) return RRN_ERR_CONFIG;
            Launch t = l;
            t.stages = S;
            t.smem = static_cast<int>(S * slot);
            ring_occ = occupancy_ln(true, dtype, add_grad, t);
            if (ring_occ < 1) return RRN_ERR_CONFIG;
            l.stages = S;
            l.smem = static_cast<int>(S * slot);
        }
    } else if (l.variant == RRN_VARIANT_ROW_WARP) {
        // a row per warp; the CTA's warps add their dw and db sums in 2 N floats of shared memory
        if (!vec_ok) return RRN_ERR_CONFIG;
        st = warp_row_layout(nvec, cfg, &l);
        if (st != RRN_OK) return st;
        l.smem = static_cast<int>(2 * N * static_cast<int64_t>(sizeof(float)));
    } else if (l.variant == RRN_VARIANT_STREAM) {
        l.vpt = 1;
        const int64_t chunks = l.vec ? nvec : N;
        l.threads = cfg && cfg->threads ? cfg->threads : (chunks >= 512 ? 512 : round_up32(chunks));
        if (l.threads < 32 || l.threads % 32 || l.threads > 1024) return RRN_ERR_CONFIG;
    } else {
        return RRN_ERR_CONFIG;
    }
    int64_t want = cfg && cfg->ctas ? cfg->ctas : 0;
    if (!want) {
        const int occ = ring_occ ? ring_occ : occupancy_ln(true, dtype, add_grad, l);
        want = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
    }
    if (want < 1) return RRN_ERR_CONFIG;
    l.ctas = M == 0 ? 0 : clamp_grid(want < M ? want : M);
    *rows_per_cta = M == 0 ? 0 : (M + l.ctas - 1) / l.ctas;
    *out = l;
    return RRN_OK;
}

int run_ln_fwd(const void *x, const void *res, void *res_out, const void *w, const void *b,
               void *y, float *mean, float *rstd, int64_t M, int64_t N, float eps, int dtype,
               const rrn_launch *cfg, cudaStream_t stream) {
    int st = check_fwd(x, res, res_out, w, y, rstd, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return RRN_OK;
    if ((b && !aligned(b, elem_size(dtype))) || (mean && !aligned(mean, 4))) return RRN_ERR_ALIGN;
    Launch l;
    st = plan_ln_fwd(vec_path_ok({x, res, res_out, w, b, y}, N, dtype), res != nullptr, M, N, dtype,
                     cfg, &l);
    if (st != RRN_OK) return st;
    LnFwdArgs a{x, res, res ? res_out : nullptr, w, b, y, mean, rstd, M, static_cast<int>(N), eps};
    cudaError_t e = dtype == RRN_BF16 ? launch_ln_fwd_bf16(a, l, stream) : launch_ln_fwd_f32(a, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

int run_ln_bwd(const void *dy, const void *d_ro, const void *x, const void *w, const float *mean,
               const float *rstd, void *dx, float *dw, float *db, void *workspace,
               size_t workspace_bytes, int64_t M, int64_t N, float eps, int dtype,
               const rrn_launch *cfg, cudaStream_t stream) {
    int st = check_bwd(dy, d_ro, x, w, rstd, dx, dw, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return zero_sums(dw, db, N, stream);
    if (!mean) return RRN_ERR_NULL;
    if (!aligned(mean, 4) || (db && !aligned(db, 4))) return RRN_ERR_ALIGN;
    Launch l;
    int64_t rpc = 0;
    st = plan_ln_bwd(vec_path_ok({dy, d_ro, x, w, dx}, N, dtype), d_ro != nullptr, M, N, dtype, cfg,
                     &l, &rpc);
    if (st != RRN_OK) return st;
    const size_t need = 2 * static_cast<size_t>(bwd_partial_rows(l)) * static_cast<size_t>(N) * sizeof(float);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return RRN_ERR_WORKSPACE;
    unsigned int *faults = nullptr;
    st = fault_word(&faults);
    if (st != RRN_OK) return st;
    LnBwdArgs a{dy, d_ro, x, w, mean, rstd, dx, dw, db, static_cast<float *>(workspace), M,
                static_cast<int>(N), 0, faults};
    cudaError_t e = dtype == RRN_BF16 ? launch_ln_bwd_bf16(a, l, stream) : launch_ln_bwd_f32(a, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

// ---------------------------------------------------------------- RMSNorm -> fp8
// The launch of the RMSNorm -> fp8 forward (rmsnorm_fwd_fp8): as the forward's planner.
int plan_quant(bool vec_ok, bool fused, int64_t M, int64_t N, int dtype, const rrn_launch *cfg,
               Launch *out) {
    const int64_t nvec = N / (16 / elem_size(dtype));
    int sms = 0;
    int st = current_sm_count(&sms);
    if (st != RRN_OK) return st;
    Launch l{};
    l.variant = cfg && cfg->variant ? cfg->variant : RRN_VARIANT_AUTO;
    if (l.variant == RRN_VARIANT_AUTO) {
        // as the forward: one row per warp for short rows over many rows (bf16 with a residual,
        // 64 Mi elements, back to back: 512 columns 198.1 -> 74.3 us, 1024 110.0 -> 71.7, 2048
        // 77.4 -> 72.1 against a row per CTA), one row per CTA while the CTA holds it, wider rows
        // split over a cluster, wider still the two-pass kernel
        const int64_t cta_max = M < 2LL * sms || !fused ? kRowCtaMaxVec : 128 * kMaxVpt;
        l.variant = !vec_ok                                  ? RRN_VARIANT_STREAM
                    : nvec <= kQuantWarpMaxVec && M >= 4LL * sms ? RRN_VARIANT_ROW_WARP
                    : nvec <= cta_max                        ? RRN_VARIANT_ROW_CTA
                    : nvec <= 2 * kClusterMaxVec             ? RRN_VARIANT_ROW_CLUSTER
                                                             : RRN_VARIANT_STREAM;
    }
    l.vec = l.variant == RRN_VARIANT_STREAM ? vec_ok : true;
    auto occ = [&](const Launch &t) {
        return dtype == RRN_BF16 ? occupancy_quant_bf16(fused, t) : occupancy_quant_f32(fused, t);
    };
    if (l.variant == RRN_VARIANT_ROW_CTA) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        st = pick_row_layout(nvec, M, sms, cfg, kMaxVpt, fwd_threads_limit, kFwdTargetThreads, &l);
        if (st != RRN_OK) return st;
        l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid(M);
    } else if (l.variant == RRN_VARIANT_ROW_WARP) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        st = warp_row_layout(nvec, cfg, &l);
        if (st != RRN_OK) return st;
        l.ctas = cfg && cfg->ctas ? cfg->ctas : clamp_grid((M + l.threads / 32 - 1) / (l.threads / 32));
    } else if (l.variant == RRN_VARIANT_ROW_CLUSTER) {
        if (!vec_ok) return RRN_ERR_CONFIG;
        // chunks above 512 vectors: 256-thread CTAs (4096 x 65536 bf16 with a residual: 294 us
        // at 4 x 256 against 432 at 8 x 128), above 1024: 512 (rows up to 16384 vectors, twice
        // the forward's limit: 2048 x 131072 357 us at 4 x 512, 516 at 8 x 256, 460 two-pass)
        const int64_t chunk = (nvec + kMaxCluster - 1) / kMaxCluster;
        const int target = chunk > 2 * kClusterChunkVec ? 512 : chunk > kClusterChunkVec ? 256 : kFwdTargetThreads;
        st = fwd_cluster_layout(nvec, M, fused, cfg, occ, &l, target);
        if (st != RRN_OK) return st;
    } else if (l.variant == RRN_VARIANT_STREAM) {
        l.vpt = 1;
        const int64_t chunks = l.vec ? nvec : N;
        // as the forward's two-pass kernel: 1024 threads from 8192 chunks a row (4096 x 65536
        // bf16 with a residual: 395 us vs 446 at 512)
        l.threads = cfg && cfg->threads ? cfg->threads
                                        : (chunks >= 8192 ? 1024 : chunks >= 512 ? 512 : round_up32(chunks));
        if (l.threads < 32 || l.threads % 32 || l.threads > 1024) return RRN_ERR_CONFIG;
        if (cfg && cfg->ctas) {
            l.ctas = cfg->ctas;
        } else {
            const int n = occ(l);
            const int64_t cap = static_cast<int64_t>(sms) * (n > 0 ? n : 1);
            l.ctas = clamp_grid(M < cap ? M : cap);
        }
    } else {
        return RRN_ERR_CONFIG;
    }
    *out = l;
    return RRN_OK;
}

int run_quant(const void *x, const void *res, void *res_out, const void *w, void *q, float *scale,
              float *rstd, int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
              cudaStream_t stream) {
    int st = check_fwd(x, res, res_out, w, x, rstd, M, N, eps, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) return RRN_OK;
    if (!q || !scale) return RRN_ERR_NULL;
    if (!aligned(scale, 4)) return RRN_ERR_ALIGN;
    const bool fused = res != nullptr;
    Launch l{};
    st = plan_quant(vec_path_ok({x, res, res_out, w, q}, N, dtype), fused, M, N, dtype, cfg, &l);
    if (st != RRN_OK) return st;
    unsigned int *faults = nullptr;
    st = fault_word(&faults);
    if (st != RRN_OK) return st;
    QuantArgs a{x, res, fused ? res_out : nullptr, w, q, scale, rstd, M, static_cast<int>(N), eps,
                faults};
    cudaError_t e = dtype == RRN_BF16 ? launch_quant_bf16(a, l, stream) : launch_quant_f32(a, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

void to_public(const Launch &l, rrn_launch *out) {
    out->variant = l.variant;
    out->vpt = l.vpt;
    out->threads = l.threads;
    out->ctas = l.ctas;
    out->stages = l.stages;
    out->cluster = l.cluster;
    out->vec = l.vec ? 1 : 0;
}

}  // namespace

int validate_bwd(const void *dy, const void *x, const void *w, const float *rstd, const void *dx,
                 const float *dw, int64_t M, int64_t N, float eps, int dtype) {
    return check_bwd(dy, nullptr, x, w, rstd, dx, dw, M, N, eps, dtype);
}

cudaError_t allow_dynamic_smem(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_pair(dev, kernel);
    std::lock_guard<std::mutex> g(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

int max_active_clusters(const void *kernel, const Launch &l) {
    if (l.cluster < 1) return 0;
    if (l.smem > 0 && allow_dynamic_smem(kernel, l.smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.cluster));
    cfg.blockDim = dim3(static_cast<unsigned>(l.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(l.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rrn

using namespace rrn;

extern "C" {

RRN_API int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd, int64_t M, int64_t N,
                        float eps, int dtype, rrn_stream_t stream) {
    return run_fwd(x, nullptr, nullptr, w, y, rstd, M, N, eps, dtype, nullptr,
                   reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_rmsnorm_fwd(const void *x, const void *residual, void *residual_out, const void *w,
                            void *y, float *rstd, int64_t M, int64_t N, float eps, int dtype,
                            rrn_stream_t stream) {
    if (!residual && M != 0) return RRN_ERR_NULL;  // (with M == 0 nothing is examined)
    return run_fwd(x, residual, residual_out, w, y, rstd, M, N, eps, dtype, nullptr,
                   reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_rmsnorm_fwd_ex(const void *x, const void *residual, void *residual_out,
                               const void *w, void *y, float *rstd, int64_t M, int64_t N,
                               float eps, int dtype, const rrn_launch *cfg, rrn_stream_t stream) {
    return run_fwd(x, residual, residual_out, w, y, rstd, M, N, eps, dtype, cfg,
                   reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes) {
    if (!bytes) return RRN_ERR_NULL;
    int st = check_common(M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) {
        *bytes = 0;
        return RRN_OK;
    }
    // The caller's buffers are not known here: size for the 128-bit vector plan and the
    // element-wise plan (unaligned buffers), plain and fused, and return the largest.
    int rows = 0;
    const bool vec_possible = N % (16 / elem_size(dtype)) == 0;
    for (int vec = 0; vec < (vec_possible ? 2 : 1); ++vec)
        for (int add = 0; add < 2; ++add) {
            Launch l;
            int64_t rpc = 0;
            st = plan_bwd_impl(vec != 0, add != 0, M, N, dtype, nullptr, &l, &rpc);
            if (st != RRN_OK) return st;
            if (bwd_partial_rows(l) > rows) rows = bwd_partial_rows(l);
        }
    *bytes = static_cast<size_t>(rows) * static_cast<size_t>(N) * sizeof(float);
    return RRN_OK;
}

RRN_API int rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd, void *dx,
                        float *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                        float eps, int dtype, rrn_stream_t stream) {
    return run_bwd(dy, nullptr, x, w, rstd, dx, dw, workspace, workspace_bytes, M, N, eps, dtype,
                   nullptr, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int rmsnorm_bwd_ex(const void *dy, const void *x, const void *w, const float *rstd,
                           void *dx, float *dw, void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                           rrn_stream_t stream) {
    return run_bwd(dy, nullptr, x, w, rstd, dx, dw, workspace, workspace_bytes, M, N, eps, dtype,
                   cfg, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_rmsnorm_bwd(const void *dy, const void *d_residual_out, const void *residual_out,
                            const void *w, const float *rstd, void *d_r, float *dw,
                            void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                            float eps, int dtype, rrn_stream_t stream) {
    return run_bwd(dy, d_residual_out, residual_out, w, rstd, d_r, dw, workspace, workspace_bytes,
                   M, N, eps, dtype, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_rmsnorm_bwd_ex(const void *dy, const void *d_residual_out,
                               const void *residual_out, const void *w, const float *rstd,
                               void *d_r, float *dw, void *workspace, size_t workspace_bytes,
                               int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                               rrn_stream_t stream) {
    return run_bwd(dy, d_residual_out, residual_out, w, rstd, d_r, dw, workspace, workspace_bytes,
                   M, N, eps, dtype, cfg, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int rrn_plan_fwd(const void *x, const void *residual, const void *residual_out,
                         const void *w, const void *y, int64_t M, int64_t N, int dtype,
                         rrn_launch *out) {
    if (!out) return RRN_ERR_NULL;
    int st = check_fwd(x, residual, residual_out, w, y, nullptr, M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    Launch l;
    st = plan_fwd_impl(vec_path_ok({x, residual, residual_out, w, y}, N, dtype), residual != nullptr,
                       M, N, dtype, nullptr, &l);
    if (st != RRN_OK) return st;
    to_public(l, out);
    return RRN_OK;
}

RRN_API int rrn_plan_bwd(const void *dy, const void *d_residual_out, const void *x,
                         const void *w, const void *dx, int64_t M, int64_t N, int dtype,
                         rrn_launch *out) {
    if (!out) return RRN_ERR_NULL;
    int st = check_common(M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    if (!dy || !x || !w || !dx) return RRN_ERR_NULL;
    Launch l;
    int64_t rpc = 0;
    st = plan_bwd_impl(vec_path_ok({dy, d_residual_out, x, w, dx}, N, dtype),
                       d_residual_out != nullptr, M, N, dtype, nullptr, &l, &rpc);
    if (st != RRN_OK) return st;
    to_public(l, out);
    return RRN_OK;
}

RRN_API int rrn_plan_layernorm_fwd(const void *x, const void *residual, const void *residual_out,
                                   const void *w, const void *b, const void *y, int64_t M, int64_t N,
                                   int dtype, rrn_launch *out) {
    if (!out) return RRN_ERR_NULL;
    int st = check_fwd(x, residual, residual_out, w, y, nullptr, M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    Launch l;
    st = plan_ln_fwd(vec_path_ok({x, residual, residual_out, w, b, y}, N, dtype), residual != nullptr, M,
                     N, dtype, nullptr, &l);
    if (st != RRN_OK) return st;
    to_public(l, out);
    return RRN_OK;
}

RRN_API int rrn_plan_layernorm_bwd(const void *dy, const void *d_residual_out, const void *x,
                                   const void *w, const void *dx, int64_t M, int64_t N, int dtype,
                                   rrn_launch *out) {
    if (!out) return RRN_ERR_NULL;
    int st = check_common(M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    if (!dy || !x || !w || !dx) return RRN_ERR_NULL;
    Launch l;
    int64_t rpc = 0;
    st = plan_ln_bwd(vec_path_ok({dy, d_residual_out, x, w, dx}, N, dtype), d_residual_out != nullptr, M,
                     N, dtype, nullptr, &l, &rpc);
    if (st != RRN_OK) return st;
    to_public(l, out);
    return RRN_OK;
}

RRN_API int rrn_plan_fwd_fp8(const void *x, const void *residual, const void *residual_out,
                             const void *w, const void *q, int64_t M, int64_t N, int dtype,
                             rrn_launch *out) {
    if (!out) return RRN_ERR_NULL;
    int st = check_fwd(x, residual, residual_out, w, x, nullptr, M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    if (!q) return RRN_ERR_NULL;
    Launch l;
    st = plan_quant(vec_path_ok({x, residual, residual_out, w, q}, N, dtype), residual != nullptr, M, N,
                    dtype, nullptr, &l);
    if (st != RRN_OK) return st;
    to_public(l, out);
    return RRN_OK;
}

RRN_API int layernorm_fwd(const void *x, const void *w, const void *b, void *y, float *mean,
                          float *rstd, int64_t M, int64_t N, float eps, int dtype,
                          rrn_stream_t stream) {
    return run_ln_fwd(x, nullptr, nullptr, w, b, y, mean, rstd, M, N, eps, dtype, nullptr,
                      reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_layernorm_fwd(const void *x, const void *residual, void *residual_out,
                              const void *w, const void *b, void *y, float *mean, float *rstd,
                              int64_t M, int64_t N, float eps, int dtype, rrn_stream_t stream) {
    if (!residual && M != 0) return RRN_ERR_NULL;  // (with M == 0 nothing is examined)
    return run_ln_fwd(x, residual, residual_out, w, b, y, mean, rstd, M, N, eps, dtype, nullptr,
                      reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int add_layernorm_fwd_ex(const void *x, const void *residual, void *residual_out,
                                 const void *w, const void *b, void *y, float *mean, float *rstd,
                                 int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                                 rrn_stream_t stream) {
    return run_ln_fwd(x, residual, residual_out, w, b, y, mean, rstd, M, N, eps, dtype, cfg,
                      reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int layernorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes) {
    if (!bytes) return RRN_ERR_NULL;
    int st = check_common(M, N, 0.f, dtype);
    if (st != RRN_OK) return st;
    if (M == 0) {
        *bytes = 0;
        return RRN_OK;
    }
    int rows = 0;
    const bool vec_possible = N % (16 / elem_size(dtype)) == 0;
    for (int vec = 0; vec < (vec_possible ? 2 : 1); ++vec)
        for (int add = 0; add < 2; ++add) {
            Launch l;
            int64_t rpc = 0;
            st = plan_ln_bwd(vec != 0, add != 0, M, N, dtype, nullptr, &l, &rpc);
            if (st != RRN_OK) return st;
            if (bwd_partial_rows(l) > rows) rows = bwd_partial_rows(l);
        }
    *bytes = 2 * static_cast<size_t>(rows) * static_cast<size_t>(N) * sizeof(float);
    return RRN_OK;
}

RRN_API int layernorm_bwd(const void *dy, const void *d_residual_out, const void *x,
                          const void *w, const float *mean, const float *rstd, void *dx,
                          float *dw, float *db, void *workspace, size_t workspace_bytes,
                          int64_t M, int64_t N, float eps, int dtype, rrn_stream_t stream) {
    return run_ln_bwd(dy, d_residual_out, x, w, mean, rstd, dx, dw, db, workspace, workspace_bytes,
                      M, N, eps, dtype, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int layernorm_bwd_ex(const void *dy, const void *d_residual_out, const void *x,
                             const void *w, const float *mean, const float *rstd, void *dx,
                             float *dw, float *db, void *workspace, size_t workspace_bytes,
                             int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                             rrn_stream_t stream) {
    return run_ln_bwd(dy, d_residual_out, x, w, mean, rstd, dx, dw, db, workspace, workspace_bytes,
                      M, N, eps, dtype, cfg, reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int rmsnorm_fwd_fp8(const void *x, const void *residual, void *residual_out,
                            const void *w, void *q, float *scale, float *rstd, int64_t M,
                            int64_t N, float eps, int dtype, rrn_stream_t stream) {
    return run_quant(x, residual, residual_out, w, q, scale, rstd, M, N, eps, dtype, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

RRN_API int rmsnorm_fwd_fp8_ex(const void *x, const void *residual, void *residual_out,
                               const void *w, void *q, float *scale, float *rstd, int64_t M,
                               int64_t N, float eps, int dtype, const rrn_launch *cfg,
                               rrn_stream_t stream) {
    return run_quant(x, residual, residual_out, w, q, scale, rstd, M, N, eps, dtype, cfg,
                     reinterpret_cast<cudaStream_t>(stream));
}

RRN_API const char *rrn_status_string(int status) {
    switch (status) {
        case RRN_OK: return "success";
        case RRN_ERR_NULL: return "a required pointer is NULL";
        case RRN_ERR_SHAPE: return "invalid shape: need M >= 0, 1 <= N <= INT32_MAX, M*N bounded";
        case RRN_ERR_EPS: return "eps must be finite and >= 0";
        case RRN_ERR_DTYPE: return "dtype must be RRN_BF16 or RRN_F32";
        case RRN_ERR_ALIGN: return "a pointer is not aligned to its element size";
        case RRN_ERR_WORKSPACE: return "workspace is NULL, unaligned or smaller than required";
        case RRN_ERR_CUDA: return "a CUDA call or kernel launch failed (see rrn_last_cuda_error)";
        case RRN_ERR_CONFIG: return "the launch configuration cannot run this problem";
        case RRN_ERR_SCRATCH: return "the problem needs more than the built-in scratch array holds";
        default: return "unknown status";
    }
}

RRN_API int rrn_last_cuda_error(void) { return t_last_cuda_error; }

RRN_API int rrn_selftest_wait_timeout(uint64_t limit_ns, rrn_stream_t stream) {
    if (limit_ns < 1000000ull) limit_ns = 1000000ull;
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    unsigned int *faults = nullptr;
    int st = fault_word(&faults);
    if (st != RRN_OK) return st;
    selftest_wait_timeout_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, faults);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return RRN_OK;
}

RRN_API int rrn_device_faults(unsigned int *faults, int clear) {
    if (!faults) return RRN_ERR_NULL;
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_faults, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e);
    if (clear && v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_faults, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *faults = v;
    return RRN_OK;
}

}  // extern "C"
