// Host-side interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rrn.h"

namespace rrn {

// Arguments of one forward call (fused when res != nullptr).
struct FwdArgs {
    const void *x;
    const void *res;  // nullptr: plain RMSNorm
    void *res_out;    // ignored when res == nullptr
    const void *w;
    void *y;
    float *rstd;      // may be nullptr
    int64_t M;
    int N;
    float eps;
    int stages;              // shared-memory ring depth (TMA variant)
    unsigned int *faults;    // the library's device fault word
};

// Arguments of one backward call. `partial` is the [P, N] fp32 workspace (P = ctas; CTA p
// handles rows p, p + P, ...).
// d_ro (nullable) is the gradient arriving at residual_out in the fused op; it is added to dx.
struct BwdArgs {
    const void *dy;
    const void *d_ro;
    const void *x;
    const void *w;
    const float *rstd;
    void *dx;
    float *dw;
    float *partial;
    int64_t M;
    int N;
    int stages;              // shared-memory ring depth (TMA variant)
    unsigned int *faults;    // the library's device fault word
};

// Arguments of one LayerNorm forward call (fused when res != nullptr; b may be nullptr).
struct LnFwdArgs {
    const void *x;
    const void *res;
    void *res_out;
    const void *w;
    const void *b;
    void *y;
    float *mean;  // may be nullptr
    float *rstd;  // may be nullptr
    int64_t M;
    int N;
    float eps;
};

// Arguments of one LayerNorm backward call. `partial` is the [2, P, N] fp32 workspace: dw
// partials in the first half, db partials in the second. d_ro and db may be nullptr.
struct LnBwdArgs {
    const void *dy;
    const void *d_ro;
    const void *x;
    const void *w;
    const float *mean;
    const float *rstd;
    void *dx;
    float *dw;
    float *db;
    float *partial;
    int64_t M;
    int N;
    int stages;             // TMA variant: ring depth
    unsigned int *faults;   // device fault word (TMA variant's bounded waits)
};

// Arguments of one RMSNorm -> fp8 e4m3 call (fused when res != nullptr).
struct QuantArgs {
    const void *x;
    const void *res;
    void *res_out;
    const void *w;
    void *q;        // [M, N] e4m3 codes
    float *scale;   // [M]
    float *rstd;    // may be nullptr
    int64_t M;
    int N;
    float eps;
    unsigned int *faults;  // the library's device fault word (cluster exchanges' bounded waits)
};

// A resolved launch (all fields set).
struct Launch {
    int variant;  // rrn_variant, never AUTO here
    int vpt;
    int threads;
    int ctas;
    bool vec;     // 128-bit vectors (else element-wise)
    int stages;   // TMA variant: rows in flight per CTA (shared-memory ring depth)
    int smem;     // dynamic shared memory bytes per CTA
    int cluster;  // CTAs per thread-block cluster (0: no cluster). Forward cluster variant: one
                  // row split across them; backward: dw partial sums pre-reduced across them.
};

// Largest vectors-per-thread the register variants are compiled for, and the thread limit
// each VPT is compiled with (__launch_bounds__), which bounds registers per thread.
constexpr int kMaxVpt = 8;
constexpr int fwd_max_threads(int vpt) { return vpt >= 8 ? 256 : vpt >= 4 ? 512 : 1024; }
// Registers per thread the row-per-CTA forward kernels may use (__maxnreg__): with VPT vectors
// per thread they launch with at most fwd_max_threads(VPT) threads, and the cap keeps that many
// resident (VPT <= 2: 48 x 1024, VPT 4: 96 x 512, VPT 8: 192 x 256 - all at most 48K of the
// SM's 64K).
constexpr int fwd_max_regs(int vpt) { return vpt <= 2 ? 48 : vpt == 4 ? 96 : 192; }
constexpr int bwd_max_threads(int vpt) { return vpt >= 4 ? 256 : 512; }
constexpr int kBwdMaxVpt = 4;
constexpr int kReduceThreads = 512;  // dw stage-2 CTA size: 32 columns x 16 row groups
constexpr int kMaxStages = 8;        // deepest shared-memory ring of the TMA variants
constexpr int kMaxCluster = 8;       // largest (portable) thread-block cluster

// The argument checks of rmsnorm_bwd (shape, dtype, eps, and - for M > 0 - pointers and their
// alignment), without the workspace; an rrn_status (defined in api.cu).
int validate_bwd(const void *dy, const void *x, const void *w, const float *rstd, const void *dx,
                 const float *dw, int64_t M, int64_t N, float eps, int dtype);

// Enqueue `kernel` on `stream` as l describes (l.ctas CTAs of l.threads threads, l.smem bytes of
// dynamic shared memory), in thread-block clusters of `cluster` CTAs when cluster > 0.
// With `programmatic`, the kernel is launched as a programmatic dependent of the kernel before it
// on the stream: it may be scheduled while that kernel drains, overlapping its launch and CTA
// start-up with the other's tail, and it waits for that kernel to complete, memory included,
// before its first access to global memory (pdl_enter in common.cuh); after any other kind of
// predecessor the launch is an ordinary one. Callers ask for it only for grids of one CTA per row
// (many waves, or few rows) with no shared-memory ring. Measured on GB300: one-row forwards of
// few rows in a CUDA graph 2.2 -> 2.0 us per launch, 16384 x 4096 forwards back to back 82.8 ->
// 81.4 us. Grids sized to one wave of resident CTAs (the backward's stage 1, cluster and ring
// kernels) keep ordinary launches: scheduled while the previous kernel still held SMs, part of
// such a grid waited for a second wave (back to back: the fused backward 89 -> 114-118 us with a
// ring on 16384 x 4096, the split-row backward 140 -> 216 us on 8192 x 16384 bf16).
inline cudaError_t enqueue(const void *kernel, const Launch &l, int cluster, bool programmatic,
                           void **params, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.ctas));
    cfg.blockDim = dim3(static_cast<unsigned>(l.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (programmatic) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, kernel, params);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device (done once
// per kernel, device and size; defined in api.cu).
cudaError_t allow_dynamic_smem(const void *kernel, int bytes);

// Clusters of l.cluster CTAs (l.threads threads, l.smem bytes of dynamic shared memory each) of
// `kernel` that the whole GPU holds at once; 0 on error (defined in api.cu). Clusters are placed
// within one GPC, so this can be below SMs x CTAs-per-SM / l.cluster.
int max_active_clusters(const void *kernel, const Launch &l);

// Kernel launchers, one per dtype (defined in fwd_bf16.cu, fwd_f32.cu and bwd.cu). They
// enqueue on `stream` and return the cudaError_t of the launch.
cudaError_t launch_fwd_bf16(const FwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_bwd_f32(const BwdArgs &a, const Launch &l, cudaStream_t stream);

cudaError_t launch_ln_fwd_bf16(const LnFwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_ln_fwd_f32(const LnFwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_ln_bwd_bf16(const LnBwdArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_ln_bwd_f32(const LnBwdArgs &a, const Launch &l, cudaStream_t stream);
// LayerNorm occupancy: bwd selects the kernel family, flag is FUSED (fwd) or ADDG (bwd).
int occupancy_ln_bf16(bool bwd, bool flag, const Launch &l);
int occupancy_ln_f32(bool bwd, bool flag, const Launch &l);

cudaError_t launch_quant_bf16(const QuantArgs &a, const Launch &l, cudaStream_t stream);
cudaError_t launch_quant_f32(const QuantArgs &a, const Launch &l, cudaStream_t stream);
int occupancy_quant_bf16(bool fused, const Launch &l);
int occupancy_quant_f32(bool fused, const Launch &l);

// Occupancy (resident CTAs per SM) of the kernel a launch would run, with l.smem bytes of
// dynamic shared memory; for a cluster launch (l.cluster > 0) the clusters resident on the
// whole GPU instead. 0 on error.
int occupancy_fwd_bf16(bool fused, const Launch &l);
int occupancy_fwd_f32(bool fused, const Launch &l);
int occupancy_bwd_bf16(bool add_grad, const Launch &l);
int occupancy_bwd_f32(bool add_grad, const Launch &l);

}  // namespace rrn
