/*
 * rrn.h - C ABI of the GB300 (sm_103a) row-wise RMSNorm / fused residual Add + RMSNorm library.
 *
 * The operation (none of the source pages writes the formula out; this is the standard
 * definition of the op they name - the RMSNorm op of the Machete page, section "Built-In
 * Areas"; the "RMSNorm SM100" example of the CuTe DSL skill page, "Workflow 0" example index;
 * KernelAgent-Oink's "RMSNorm and fused Add + RMSNorm" custom ops, KernelAgent page,
 * repository summary), per row i of an [M, N] row-major matrix:
 *
 *     r_i    = x_i + residual_i                 (fused op; written back as residual_out)
 *     rstd_i = 1 / sqrt( mean_j(r_ij^2) + eps )
 *     y_ij   = r_ij * rstd_i * w_j
 *
 * and the backward pass of the plain op (x -> y), with xhat = x * rstd and g = dy * w:
 *
 *     dx_ij = rstd_i * ( g_ij - xhat_ij * mean_k(g_ik * xhat_ik) )
 *     dw_j  = sum_i dy_ij * xhat_ij
 *
 * Arithmetic: inputs are widened to fp32; the sum of squares (and the backward dot product)
 * is accumulated in fp32 with warp shuffles followed by a cross-warp shared-memory step (the
 * reduction pattern the CuTe DSL skill page prescribes for RMSNorm: "Workflow 0", paragraph on
 * reduction kernels); y is computed from the UNROUNDED fp32 r and rounded once (round to
 * nearest even) to the storage type. residual_out is r rounded once to the storage type.
 * dw is reduced in two stages in a fixed order, so it is bitwise reproducible for a given
 * (M, N, dtype, device).
 *
 * Conventions shared by every entry point below:
 *   - Pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors) on the current device,
 *     except where stated. The caller owns every buffer; the library allocates nothing,
 *     never synchronises and compiles nothing at run time.
 *   - Layout: x, residual, residual_out, y, dy, dx are contiguous row-major [M, N] (row stride
 *     N elements) of `dtype`; w is [N] of `dtype`; rstd is [M] fp32; dw is [N] fp32.
 *   - dtype: RRN_BF16 (bfloat16) or RRN_F32 (float); all dtype-typed tensors of a call share it.
 *   - Alignment: elements must be naturally aligned (2 bytes for bf16, 4 for fp32; rstd and
 *     dw 4 bytes). When every matrix pointer is 16-byte aligned and N * sizeof(dtype) is a
 *     multiple of 16 the 128-bit vector kernels run; otherwise an element-wise GPU kernel
 *     runs. There is no CPU fallback.
 *   - Aliasing: an output may be the same buffer as an input of the same shape
 *     (residual_out == residual or x; y == x; dx == dy or x; d_r == dy, d_residual_out or
 *     residual_out). Any other overlap is undefined.
 *   - M == 0 returns RRN_OK after dtype, N and eps are checked. The forward calls then launch
 *     nothing and examine no pointer (all may be NULL). The backward calls read no row either,
 *     but dw (and db) are sums over no rows: they are set to zero on `stream`, so dw (and db,
 *     where given) must then be valid, 4-byte aligned device pointers; the other pointers and
 *     the workspace are not examined.
 *   - Work is enqueued on `stream` (NULL: the legacy default stream) and the call returns
 *     without waiting. Argument errors return a nonzero code before anything is launched;
 *     a failed launch returns RRN_ERR_CUDA (rrn_last_cuda_error() gives the cudaError_t);
 *     errors during execution surface on the stream like any CUDA error.
 *   - Thread safety: every entry point may be called from several host threads at once.
 */
#ifndef RRN_H_
#define RRN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RRN_API __attribute__((visibility("default")))
#else
#define RRN_API
#endif

/* A CUDA stream handle: the same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *rrn_stream_t;

/* Storage types. */
typedef enum { RRN_BF16 = 0, RRN_F32 = 1 } rrn_dtype;

/* Return codes. */
typedef enum {
    RRN_OK = 0,
    RRN_ERR_NULL = 1,      /* a required pointer is NULL */
    RRN_ERR_SHAPE = 2,     /* M < 0, N < 1, or M * N too large */
    RRN_ERR_EPS = 3,       /* eps negative, infinite or NaN */
    RRN_ERR_DTYPE = 4,     /* dtype not RRN_BF16 / RRN_F32 */
    RRN_ERR_ALIGN = 5,     /* a pointer is not aligned to its element size */
    RRN_ERR_WORKSPACE = 6, /* backward workspace NULL or smaller than required */
    RRN_ERR_CUDA = 7,      /* a CUDA runtime call or kernel launch failed */
    RRN_ERR_CONFIG = 8,    /* an explicit launch configuration cannot cover the row */
    RRN_ERR_SCRATCH = 9    /* the problem needs more than the built-in scratch array holds */
} rrn_status;

/*
 * rmsnorm_fwd - RMSNorm forward: y = x * rstd * w per row (Machete page, "Built-In Areas").
 *   x     [M, N] dtype, read.
 *   w     [N] dtype, read.
 *   y     [M, N] dtype, written (may be x).
 *   rstd  [M] fp32, written; may be NULL (not stored).
 *   eps   >= 0, finite; added to the mean square inside the square root.
 * Returns an rrn_status.
 */
RRN_API int rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd, int64_t M, int64_t N,
                        float eps, int dtype, rrn_stream_t stream);

/*
 * add_rmsnorm_fwd - fused residual Add + RMSNorm forward (KernelAgent page, repository
 * summary: KernelAgent-Oink's "fused Add + RMSNorm"): r = x + residual in fp32,
 * residual_out = r (rounded to dtype), y = r * rstd * w (from the unrounded r).
 *   x, residual   [M, N] dtype, read.
 *   residual_out  [M, N] dtype, written (may be residual or x: the in-place update).
 *   w             [N] dtype, read.
 *   y             [M, N] dtype, written.
 *   rstd          [M] fp32, written; may be NULL.
 * Returns an rrn_status.
 */
RRN_API int add_rmsnorm_fwd(const void *x, const void *residual, void *residual_out, const void *w,
                            void *y, float *rstd, int64_t M, int64_t N, float eps, int dtype,
                            rrn_stream_t stream);

/*
 * rmsnorm_bwd_workspace_bytes - device workspace rmsnorm_bwd needs for (M, N, dtype) on the
 * CURRENT device (it depends on the device's SM count). Writes the size to *bytes (0 when
 * M == 0). Returns an rrn_status (RRN_ERR_CUDA if the device cannot be queried).
 */
RRN_API int rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes);

/*
 * rmsnorm_bwd - RMSNorm backward of rmsnorm_fwd, with a two-stage deterministic dw: the
 * gradients of the Machete page's RMSNorm op (section "Built-In Areas", which lists autograd
 * helpers beside the ops). The pages write no backward formula; the one at the top of this
 * file is the exact derivative of the forward definition (d rstd / d x_k = -rstd^3 x_k / N),
 * dx plus a dw summed over the rows.
 *   dy        [M, N] dtype, read (upstream gradient of y).
 *   x         [M, N] dtype, read (the forward input).
 *   w         [N] dtype, read.
 *   rstd      [M] fp32, read (as written by the forward pass).
 *   dx        [M, N] dtype, written (may be dy or x).
 *   dw        [N] fp32, overwritten (not accumulated) with the sum over all M rows.
 *   workspace device buffer of at least rmsnorm_bwd_workspace_bytes(M, N, dtype) bytes,
 *             16-byte aligned, owned by the caller; its contents on entry are ignored and
 *             on return are unspecified. Calls that share a workspace must be ordered on
 *             one stream.
 *   eps       validated (>= 0, finite) and otherwise unused: rstd carries it.
 * Stage 1 writes per-CTA fp32 partial sums of dy * xhat to the workspace; stage 2 adds
 * them in a fixed order. With M == 0 dw is set to zero (an empty sum) and no workspace is used.
 * Returns an rrn_status.
 */
RRN_API int rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd, void *dx,
                        float *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                        float eps, int dtype, rrn_stream_t stream);

/*
 * rmsnorm_bwd_noalloc - rmsnorm_bwd without a caller-provided workspace, for callers that
 * cannot allocate device memory: plugins inside an engine that owns every device allocation and
 * hands a plugin only its inputs and outputs, and C callers without a caching allocator, for whom
 * a cudaMalloc/cudaFree pair per call would synchronise the device. (The source pages have no
 * counterpart of this entry point; it is a deployment convenience of this library.)
 *   Arguments, layout and error codes as for rmsnorm_bwd, without the workspace arguments; the
 *   argument checks run first, and M == 0 sets dw to zero as rmsnorm_bwd does.
 *   The dw partial sums live in one 8 MiB array of fp32 inside the library (a __device__
 *   variable, held by every GPU that loads the library until the process exits). The stage-1
 *   launch is rmsnorm_bwd's, with the rows of partial sums it writes (one per CTA, or one per
 *   cluster when each row is split over a cluster) lowered until rows * N <= 2,097,152;
 *   N > 2,097,152 returns RRN_ERR_SCRATCH.
 *   Determinism: dw is bitwise reproducible from one rmsnorm_bwd_noalloc call to the next (same
 *   M, N, dtype and device). Where the rows of partial sums had to be lowered, the sums are
 *   added in another order than rmsnorm_bwd adds them, so dw can differ from rmsnorm_bwd's in
 *   the last bits (within the dw tolerance); dx is the same.
 *   Nothing in the array needs to start at zero (stage 1 writes all that stage 2 reads).
 *   All calls on a device share the array: calls whose kernels overlap on the GPU race - order
 *   them on one stream. The first call on each device looks the array's address up through the
 *   CUDA runtime (with that device current); later calls on that device reuse it.
 *   No cudaMalloc, cudaFree or other allocation happens. Returns an rrn_status.
 */
RRN_API int rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *w, const float *rstd,
                                void *dx, float *dw, int64_t M, int64_t N, float eps, int dtype,
                                rrn_stream_t stream);

/*
 * add_rmsnorm_bwd - backward of the fused residual Add + RMSNorm (add_rmsnorm_fwd), in one pass:
 *   d_r = d_residual_out + rstd * (g - rhat * mean(g * rhat)),  g = dy * w,  rhat = r * rstd
 *   dw  = sum over rows of dy * rhat
 * where r is the forward's residual_out as stored. d_r is the gradient with respect to
 * r = x + residual, i.e. with respect to both x and residual. (The backward of the KernelAgent
 * page's fused Add + RMSNorm op; Machete's "Built-In Areas" lists autograd helpers.)
 *   dy              [M, N] dtype, read (gradient arriving at y).
 *   d_residual_out  [M, N] dtype, read; may be NULL (no gradient arrives at residual_out).
 *   residual_out    [M, N] dtype, read (the forward's r).
 *   w               [N] dtype, read.
 *   rstd            [M] fp32, read (as written by the forward pass).
 *   d_r             [M, N] dtype, written (may be dy, d_residual_out or residual_out).
 *   dw, workspace   as for rmsnorm_bwd (same workspace size query).
 * Returns an rrn_status.
 */
RRN_API int add_rmsnorm_bwd(const void *dy, const void *d_residual_out, const void *residual_out,
                            const void *w, const float *rstd, void *d_r, float *dw,
                            void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                            float eps, int dtype, rrn_stream_t stream);

/*
 * LayerNorm, the mean-subtracting variant (the CuTe DSL skill page lists a "CTA norm
 * (LayerNorm)" example in its "Workflow 0" example index). Per row of r = x (+ residual):
 *     mean = mean_j(r_j),  rstd = 1 / sqrt( mean_j((r_j - mean)^2) + eps ),
 *     y_j  = (r_j - mean) * rstd * w_j + b_j
 * computed in fp32 with the variance taken about the mean (two passes over the row).
 *
 * layernorm_fwd / add_layernorm_fwd
 *   x, residual, residual_out, w, y, rstd   as for rmsnorm_fwd / add_rmsnorm_fwd.
 *   b      [N] dtype, read; may be NULL (no bias).
 *   mean   [M] fp32, written; may be NULL.
 * add_layernorm_fwd_ex takes residual == NULL for the plain op and an explicit launch
 * configuration (RRN_VARIANT_ROW_CTA or RRN_VARIANT_STREAM).
 *
 * layernorm_bwd - dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) (+ d_residual_out),
 *   g = dy * w, xhat = (x - mean) * rstd;  dw = sum_rows dy * xhat;  db = sum_rows dy.
 *   dy              [M, N] dtype, read.
 *   d_residual_out  [M, N] dtype, read; may be NULL (plain op, or no gradient at residual_out).
 *   x               [M, N] dtype, read: the forward input (the stored residual_out when fused).
 *   w               [N] dtype, read.   mean, rstd  [M] fp32, read (as the forward wrote them).
 *   dx              [M, N] dtype, written (may alias dy, d_residual_out or x).
 *   dw, db          [N] fp32, overwritten; db may be NULL.
 *   workspace       at least layernorm_bwd_workspace_bytes(M, N, dtype) bytes (twice the
 *                   RMSNorm workspace: dw and db partials), 16-byte aligned.
 * Each returns an rrn_status.
 */
RRN_API int layernorm_fwd(const void *x, const void *w, const void *b, void *y, float *mean,
                          float *rstd, int64_t M, int64_t N, float eps, int dtype,
                          rrn_stream_t stream);
RRN_API int add_layernorm_fwd(const void *x, const void *residual, void *residual_out,
                              const void *w, const void *b, void *y, float *mean, float *rstd,
                              int64_t M, int64_t N, float eps, int dtype, rrn_stream_t stream);
RRN_API int layernorm_bwd_workspace_bytes(int64_t M, int64_t N, int dtype, size_t *bytes);
RRN_API int layernorm_bwd(const void *dy, const void *d_residual_out, const void *x,
                          const void *w, const float *mean, const float *rstd, void *dx,
                          float *dw, float *db, void *workspace, size_t workspace_bytes,
                          int64_t M, int64_t N, float eps, int dtype, rrn_stream_t stream);

/*
 * rmsnorm_fwd_fp8 - RMSNorm (fused with the residual add when `residual` is not NULL) feeding an
 * FP8 E4M3 output with one fp32 scale per row, for a following FP8 GEMM - the norm fused with
 * its neighbouring op in one pass, as a persistent megakernel would do (Machete page, "Core
 * Ideas"). Per row, in fp32: y = r * rstd * w as rmsnorm_fwd computes it;
 * amax = max_j |y_j|; scale = amax / 448; q_j = e4m3(y_j * (448 / amax)), rounded to nearest
 * even with saturation to +/-448 (scale = 0 and q = 0 when y is all zero). Dequantised,
 * q_j * scale approximates y_j within half an e4m3 step.
 *   x, residual, residual_out, w, rstd   as for add_rmsnorm_fwd (residual may be NULL: plain op;
 *                                        residual_out is then ignored).
 *   q      [M, N] bytes (e4m3 codes, 0x7F/0xFF never produced), written.
 *   scale  [M] fp32, written.
 * Returns an rrn_status. rmsnorm_fwd_fp8_ex (declared with the launch-control calls below)
 * takes an explicit launch configuration (RRN_VARIANT_ROW_CTA, RRN_VARIANT_ROW_CLUSTER or
 * RRN_VARIANT_STREAM).
 */
RRN_API int rmsnorm_fwd_fp8(const void *x, const void *residual, void *residual_out,
                            const void *w, void *q, float *scale, float *rstd, int64_t M,
                            int64_t N, float eps, int dtype, rrn_stream_t stream);

/* rrn_status_string - static, NUL-terminated description of a status code. */
RRN_API const char *rrn_status_string(int status);

/* rrn_last_cuda_error - the cudaError_t behind this thread's last RRN_ERR_CUDA (0 if none). */
RRN_API int rrn_last_cuda_error(void);

/*
 * rrn_device_faults - read (and, if `clear` is nonzero, reset) the library's fault word on the
 * current device. Bit 0 (RRN_FAULT_WAIT_TIMEOUT) is set when a kernel gave up waiting for an
 * asynchronous copy (a bounded wait of about 2 s ran out); that kernel's outputs are then
 * invalid. The kernels never trap. This call synchronises with the device (it copies the
 * word), unlike every other entry point. Returns an rrn_status.
 */
#define RRN_FAULT_WAIT_TIMEOUT 1u
RRN_API int rrn_device_faults(unsigned int *faults, int clear);

/*
 * rrn_selftest_wait_timeout - exercise the bounded-wait failure path on the current device:
 * one thread waits on an mbarrier that nothing ever arrives at, gives up after `limit_ns`
 * nanoseconds (clamped to 1 ms .. 1 s), sets RRN_FAULT_WAIT_TIMEOUT in the fault word and
 * returns normally; the context stays usable. Enqueued on `stream`. Returns an rrn_status.
 */
RRN_API int rrn_selftest_wait_timeout(uint64_t limit_ns, rrn_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Launch control, for benchmarking and tuning. The entry points above choose these
 * automatically from (M, N, dtype, SM count); the _ex forms below take them explicitly.
 * ------------------------------------------------------------------------------------------ */

/* Kernel variants. */
typedef enum {
    RRN_VARIANT_AUTO = 0,    /* let the library choose */
    RRN_VARIANT_ROW_CTA = 1, /* one row per CTA, row held in registers, 128-bit vectors */
    RRN_VARIANT_ROW_WARP = 2,/* one row per warp, row held in registers, 128-bit vectors
                                (rows of at most 8 x 32 vectors; the RMSNorm, fp8 and LayerNorm
                                forwards) */
    RRN_VARIANT_STREAM = 3,  /* one row per CTA, two passes over the row (any N / alignment) */
    RRN_VARIANT_ROW_TMA = 4, /* persistent row per CTA fed by bulk async copies (TMA engine)
                                into a shared-memory ring of `stages` rows, 128-bit vectors */
    RRN_VARIANT_ROW_CLUSTER = 5 /* one row split across the `cluster` CTAs of a thread-block
                                   cluster; partial sums exchanged in distributed shared memory.
                                   RMSNorm forward and backward, the fp8 forward and the
                                   LayerNorm backward (a backward's workspace then needs one
                                   row per cluster, two for LayerNorm). */
} rrn_variant;

/* A launch configuration. Zero fields mean "choose automatically". */
typedef struct {
    int variant; /* rrn_variant */
    int vpt;     /* 128-bit vectors per thread for the register variants: 1, 2, 4 or 8 */
    int threads; /* threads per CTA (a multiple of 32, at most 1024) */
    int ctas;    /* CTAs in the grid; each walks rows with a grid-sized stride */
    int stages;  /* RRN_VARIANT_ROW_TMA: rows in flight per CTA, 1..8 (the LayerNorm
                    backward: ring slots, 2..8, holding S - 1 rows in flight) */
    int cluster; /* RRN_VARIANT_ROW_CLUSTER: CTAs per cluster, 2..8 (ctas a multiple of it).
                    Backward ROW_CTA, ROW_TMA: 2, 4 or 8 = add the dw partial sums of
                    that many stage-1 CTAs through distributed shared memory before stage 2
                    (used when there are at least twice that many CTAs; the CTA count is
                    rounded down to a multiple of it), 1 = no clusters, 0 = the planner's
                    choice (currently no clusters). */
    int vec;     /* output of rrn_plan_*: 1 when the 128-bit vector path is used */
} rrn_launch;

/*
 * rrn_plan_fwd / rrn_plan_bwd - the configuration the automatic entry points would use for
 * these arguments (the pointers only matter for their alignment; they are not dereferenced).
 * `residual` NULL plans the plain forward; `d_residual_out` NULL plans rmsnorm_bwd, non-NULL
 * add_rmsnorm_bwd (x is then residual_out and dx is d_r). Returns an rrn_status.
 */
RRN_API int rrn_plan_fwd(const void *x, const void *residual, const void *residual_out,
                         const void *w, const void *y, int64_t M, int64_t N, int dtype,
                         rrn_launch *out);
RRN_API int rrn_plan_bwd(const void *dy, const void *d_residual_out, const void *x,
                         const void *w, const void *dx, int64_t M, int64_t N, int dtype,
                         rrn_launch *out);
/*
 * rrn_plan_layernorm_fwd / rrn_plan_layernorm_bwd / rrn_plan_fwd_fp8 - the same for
 * add_layernorm_fwd (`residual` NULL: layernorm_fwd; b may be NULL), layernorm_bwd
 * (`d_residual_out` NULL: the plain backward; the stage-1 launch) and rmsnorm_fwd_fp8 (q: the
 * codes). Returns an rrn_status.
 */
RRN_API int rrn_plan_layernorm_fwd(const void *x, const void *residual, const void *residual_out,
                                   const void *w, const void *b, const void *y, int64_t M, int64_t N,
                                   int dtype, rrn_launch *out);
RRN_API int rrn_plan_layernorm_bwd(const void *dy, const void *d_residual_out, const void *x,
                                   const void *w, const void *dx, int64_t M, int64_t N, int dtype,
                                   rrn_launch *out);
RRN_API int rrn_plan_fwd_fp8(const void *x, const void *residual, const void *residual_out,
                             const void *w, const void *q, int64_t M, int64_t N, int dtype,
                             rrn_launch *out);

/*
 * add_rmsnorm_fwd_ex - add_rmsnorm_fwd (residual != NULL) or rmsnorm_fwd (residual == NULL,
 * residual_out ignored) with an explicit launch configuration `cfg` (NULL: automatic).
 * Fields left at 0 are filled in automatically; a configuration whose threads * vpt vectors
 * cannot cover a row, or that the chosen variant cannot run, returns RRN_ERR_CONFIG.
 */
RRN_API int add_rmsnorm_fwd_ex(const void *x, const void *residual, void *residual_out,
                               const void *w, void *y, float *rstd, int64_t M, int64_t N,
                               float eps, int dtype, const rrn_launch *cfg, rrn_stream_t stream);

/* rmsnorm_fwd_fp8 with an explicit launch configuration (row-per-CTA, row-per-warp, cluster
 * split or two-pass). */
RRN_API int rmsnorm_fwd_fp8_ex(const void *x, const void *residual, void *residual_out,
                               const void *w, void *q, float *scale, float *rstd, int64_t M,
                               int64_t N, float eps, int dtype, const rrn_launch *cfg,
                               rrn_stream_t stream);

/* LayerNorm with an explicit launch configuration: the forward row-per-CTA, row-per-warp or
 * two-pass; the backward row-per-CTA, two-pass, the TMA ring (ROW_TMA) and the cluster split
 * (ROW_CLUSTER; workspace: one dw and one db row per cluster). */
RRN_API int add_layernorm_fwd_ex(const void *x, const void *residual, void *residual_out,
                                 const void *w, const void *b, void *y, float *mean, float *rstd,
                                 int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                                 rrn_stream_t stream);
RRN_API int layernorm_bwd_ex(const void *dy, const void *d_residual_out, const void *x,
                             const void *w, const float *mean, const float *rstd, void *dx,
                             float *dw, float *db, void *workspace, size_t workspace_bytes,
                             int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                             rrn_stream_t stream);

/* rmsnorm_bwd_ex / add_rmsnorm_bwd_ex - the backward calls with an explicit stage-1 launch
 * configuration (see above). The workspace must hold one row of N fp32 values per stage-1 CTA,
 * or per cluster when the CTAs work in clusters (cfg->ctas / cfg->cluster rows); rrn_plan_bwd
 * reports the default configuration. */
RRN_API int rmsnorm_bwd_ex(const void *dy, const void *x, const void *w, const float *rstd,
                           void *dx, float *dw, void *workspace, size_t workspace_bytes,
                           int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                           rrn_stream_t stream);
RRN_API int add_rmsnorm_bwd_ex(const void *dy, const void *d_residual_out,
                               const void *residual_out, const void *w, const float *rstd,
                               void *d_r, float *dw, void *workspace, size_t workspace_bytes,
                               int64_t M, int64_t N, float eps, int dtype, const rrn_launch *cfg,
                               rrn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RRN_H_ */
