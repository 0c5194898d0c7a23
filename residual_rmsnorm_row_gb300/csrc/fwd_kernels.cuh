// Forward kernels: RMSNorm and fused residual Add + RMSNorm, one row at a time.
//
//   r = x (+ residual)          fp32, residual_out = RN(r)         (fused only)
//   rstd = rsqrt(sum(r^2) / N + eps)
//   y = RN(r * rstd * w)        from the unrounded fp32 r
//
// Three shapes of the same computation (the pages name the op - Machete "Built-In Areas",
// KernelAgent-Oink's RMSNorm and fused Add + RMSNorm - and, for the reduction, the
// warp-shuffle-then-shared-memory pattern of the CuTe DSL skill page; the kernels are this
// library's own design for sm_103a):
//   fwd_row_cta     one row per CTA, the row held in registers as 128-bit vectors; the grid
//                   walks rows with a grid-sized stride (persistent when the grid is smaller
//                   than M, one row per CTA when it is not). Rows up to 1024 vectors (bf16
//                   N <= 8192), up to 2048 when there are few rows.
//   fwd_row_warp    one row per warp, no barrier at all; for short rows (bf16 N <= 2048).
//   fwd_row_cluster one row split over the CTAs of a thread-block cluster (wider rows).
//   fwd_row_tma     row per CTA fed through a shared-memory ring by bulk copies (on request).
//   fwd_stream      one row per CTA in two passes over global memory (sum of squares, then
//                   normalise, re-reading the row from L2): any N and any alignment.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace rrn {

// The per-row work of the row-per-CTA variants, on a row already in registers: this thread
// owns the 128-bit vectors c = v * blockDim.x + threadIdx.x (v < VPT, c < nvec) of x (xv) and
// residual (rv). The weight vectors are read where they are used, from L1 (the kernels prefetch
// them there), rather than held in registers across rows: fewer registers per thread means
// more CTAs - more rows in flight - per SM. Writes residual_out (fused), y and rstd.
// `after_reduce` runs right after the CTA-wide sum of squares, when every thread has consumed
// its inputs; when it returns false the row is abandoned (nothing more is written).
template <typename T, int VPT, bool FUSED, typename AfterReduce>
__device__ __forceinline__ bool row_cta_body(const FwdArgs &a, int64_t row, int nvec,
                                             const uint4 (&xv)[VPT], const uint4 (&rv)[VPT],
                                             float (&slots)[2][32], int &parity,
                                             AfterReduce after_reduce) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int64_t base = row * nvec;
    const float n_f = static_cast<float>(a.N);
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float f[V];
            r_of<T, FUSED>(xv[v], rv[v], f);
            if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
#pragma unroll
            for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
        }
    }
    ss = cta_sum(ss, slots[parity]);
    parity ^= 1;
    if (!after_reduce()) return false;
    float rs;
    if (!needs_rescale(ss)) {
        rs = rstd_plain(ss, n_f, a.eps);
    } else {  // rare: sum of squares out of fp32 range, or an all-zero row
        float am = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v)
            if (v * nthr + tid < nvec) {
                float f[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(f[k]));
            }
        am = cta_max(am, slots[parity]);
        parity ^= 1;
        const int e = rescale_exponent(am);
        float s2 = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v)
            if (v * nthr + tid < nvec) {
                float f[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const float t = ldexpf(f[k], -e);
                    s2 = fmaf(t, t, s2);
                }
            }
        s2 = cta_sum(s2, slots[parity]);
        parity ^= 1;
        rs = rstd_rescaled(s2, n_f, a.eps, e);
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float f[V], wf[V], o[V];
            r_of<T, FUSED>(xv[v], rv[v], f);
            E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
#pragma unroll
            for (int k = 0; k < V; ++k) o[k] = f[k] * rs * wf[k];
            st_stream(static_cast<uint4 *>(a.y) + base + c, E::pack(o));
        }
    }
    if (tid == 0 && a.rstd) a.rstd[row] = rs;
    return true;
}

// Start pulling this thread's weight vectors into L1 (they are read after the reduction).
template <int VPT>
__device__ __forceinline__ void prefetch_w(const FwdArgs &a, int nvec) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * blockDim.x + threadIdx.x;
        if (c < nvec) prefetch_l1(static_cast<const uint4 *>(a.w) + c);
    }
}

template <typename T, int VPT, bool FUSED>
__global__ void __maxnreg__(fwd_max_regs(VPT)) fwd_row_cta(const FwdArgs a) {
    pdl_enter();
    constexpr int V = Elem<T>::kPerVec;
    __shared__ float slots[2][32];
    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    const uint4 *r4 = static_cast<const uint4 *>(a.res);
    prefetch_w<VPT>(a, nvec);

    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_stream(x4 + base + c);
                if (FUSED) rv[v] = ld_stream(r4 + base + c);
            }
        }
        row_cta_body<T, VPT, FUSED>(a, row, nvec, xv, rv, slots, parity, [] { return true; });
    }
}

// Row per CTA, persistent, fed by the TMA engine: CTA b owns rows b, b + G, b + 2G, ...
// (G = gridDim.x) and keeps a.stages of them in flight in a shared-memory ring, each row (x and,
// fused, residual) fetched by one thread with cp.async.bulk and counted on that slot's
// mbarrier. Once the CTA-wide sum of a row is done every thread holds its share of the row in
// registers, so the slot is refilled right then with the row `stages` iterations ahead.
// Bytes in flight per SM = resident CTAs x stages x row bytes, independent of registers.
template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(fwd_max_threads(VPT))
    fwd_row_tma(const FwdArgs a) {
    pdl_enter();
    constexpr int V = Elem<T>::kPerVec;
    constexpr int NT = FUSED ? 2 : 1;
    extern __shared__ __align__(128) unsigned char ring_buf[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ float slots[2][32];
    __shared__ int abort_flag;

    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    RowRing<NT> ring;
    ring.buf = ring_buf;
    ring.full = full;
    ring.src[0] = static_cast<const char *>(a.x);
    if constexpr (FUSED) ring.src[NT - 1] = static_cast<const char *>(a.res);
    ring.row_bytes = static_cast<uint32_t>(a.N) * static_cast<uint32_t>(sizeof(T));
    ring.S = a.stages;
    ring.first = blockIdx.x;
    ring.stride = gridDim.x;
    ring.nrows = ring.first < a.M ? (a.M - 1 - ring.first) / ring.stride + 1 : 0;

    if (tid == 0) {
        ring.init();
        abort_flag = 0;
    }
    __syncthreads();
    if (tid == 0) ring.prime();

    prefetch_w<VPT>(a, nvec);

    int parity = 0;
    int64_t k = 0;
    for (; k < ring.nrows; ++k) {
        if (!ring.wait(a.faults)) abort_flag = 1;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_shared_v4(ring.slot(0) + static_cast<size_t>(c) * 16);
                if (FUSED) rv[v] = ld_shared_v4(ring.slot(NT - 1) + static_cast<size_t>(c) * 16);
            }
        }
        const bool done = row_cta_body<T, VPT, FUSED>(
            a, ring.first + k * ring.stride, nvec, xv, rv, slots, parity, [&] {
                if (abort_flag) return false;  // written before the barrier: uniform
                if (tid == 0 && k + ring.S < ring.nrows) {
                    fence_proxy_async();       // our generic reads of the slot come first
                    ring.issue(k + ring.S, ring.cur);
                }
                return true;
            });
        if (!done) break;
        ring.advance();
    }
    // A wait ran out: let the copies already issued land before the CTA's shared memory is
    // released, then leave; the fault word tells the host.
    if (k < ring.nrows && tid == 0) ring.drain(k, ring.S);
}

// One row split across the C CTAs of a thread-block cluster (C = 2..8): CTA rank q owns the
// vectors [q * chunk, (q + 1) * chunk) of every row its cluster handles (chunk = ceil(nvec / C)),
// held in registers. The CTAs' partial sums of squares are exchanged through distributed shared
// memory (ClusterExchange: asynchronous remote stores counted on mbarriers, no cluster barrier per
// row) and every CTA adds the C values in rank order (the same bits everywhere). Clusters
// walk rows with a grid-sized stride. For rows too wide for one CTA's registers, and to spread
// few-row (decode) problems over more SMs.
template <typename T, int VPT, bool FUSED>
__device__ __forceinline__ void fwd_row_cluster_body(const FwdArgs &a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    __shared__ float slots[2][32];
    __shared__ float part[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    ClusterExchange<float, kMaxCluster> xchg(part, xbar);

    const int nvec = a.N / V;
    const int C = static_cast<int>(cluster_nctarank());
    const int q = static_cast<int>(cluster_ctarank());
    const int chunk = (nvec + C - 1) / C;
    const int c0 = q * chunk;
    const int c1 = min(nvec, c0 + chunk);
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    const uint4 *r4 = static_cast<const uint4 *>(a.res);
    if (tid == 0) xchg.init();
    cluster_sync();  // every CTA of the cluster runs and has its barriers initialised

    uint4 wv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
    }
    int parity = 0;
    // Cluster-wide total (or maximum) of one float per CTA; every CTA gets the same bits.
    auto exchange = [&](float mine, bool take_max) {
        return take_max ? xchg(mine, 0.f, [](float u, float v) { return fmaxf(u, v); }, a.faults)
                        : xchg(mine, 0.f, [](float u, float v) { return u + v; }, a.faults);
    };

    const int64_t ncl = cluster_nclusters_x();
    for (int64_t row = cluster_id_x(); row < a.M; row += ncl) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                xv[v] = ld_stream(x4 + base + c);
                if (FUSED) rv[v] = ld_stream(r4 + base + c);
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float f[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
#pragma unroll
                for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
            }
        }
        ss = cta_sum(ss, slots[parity]);
        parity ^= 1;
        ss = exchange(ss, false);
        float rs;
        if (!needs_rescale(ss)) {
            rs = rstd_plain(ss, n_f, a.eps);
        } else {  // rare: sum of squares out of fp32 range, or an all-zero row
            float am = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (c0 + v * nthr + tid < c1) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(f[k]));
                }
            am = cta_max(am, slots[parity]);
            parity ^= 1;
            const int e = rescale_exponent(exchange(am, true));
            float s2 = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (c0 + v * nthr + tid < c1) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float t = ldexpf(f[k], -e);
                        s2 = fmaf(t, t, s2);
                    }
                }
            s2 = cta_sum(s2, slots[parity]);
            parity ^= 1;
            rs = rstd_rescaled(exchange(s2, false), n_f, a.eps, e);
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float f[V], wf[V], o[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = f[k] * rs * wf[k];
                st_stream(static_cast<uint4 *>(a.y) + base + c, E::pack(o));
            }
        }
        if (q == 0 && tid == 0 && a.rstd) a.rstd[row] = rs;
    }
    cluster_sync();  // no CTA exits while a peer may still write into its shared memory
}

// The cluster kernel; at 8 vectors a thread compiled for 2 CTAs of 256 threads (at most 128
// registers instead of 166 with a residual, 88 bytes of it spilled to local memory: 4 CTAs of
// 128 threads per SM instead of 3; 4096 x 65536 bf16 with a residual 369.8 -> 350.3 us). Fewer
// vectors a thread keep the compiler's own allocation (the same bound there cost 6-7 % on
// 16384- and 32768-wide rows).
template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(fwd_max_threads(VPT)) fwd_row_cluster(const FwdArgs a) {
    fwd_row_cluster_body<T, VPT, FUSED>(a);
}
template <typename T, bool FUSED>
__global__ void __launch_bounds__(fwd_max_threads(8), 2) fwd_row_cluster_v8(const FwdArgs a) {
    fwd_row_cluster_body<T, 8, FUSED>(a);
}

template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(256) fwd_row_warp(const FwdArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;

    const int nvec = a.N / V;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    const uint4 *r4 = static_cast<const uint4 *>(a.res);
    uint4 *ro4 = static_cast<uint4 *>(a.res_out);
    uint4 *y4 = static_cast<uint4 *>(a.y);
    const float n_f = static_cast<float>(a.N);

    uint4 wv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * 32 + lane;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
    }

    for (int64_t row = warp0; row < a.M; row += nwarps) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                xv[v] = ld_stream(x4 + base + c);
                if (FUSED) rv[v] = ld_stream(r4 + base + c);
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                if (FUSED) st_stream(ro4 + base + c, E::pack(f));
#pragma unroll
                for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
            }
        }
        ss = warp_sum(ss);
        float rs;
        if (!needs_rescale(ss)) {
            rs = rstd_plain(ss, n_f, a.eps);
        } else {  // rare: sum of squares out of fp32 range, or an all-zero row
            float am = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * 32 + lane < nvec) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(f[k]));
                }
            const int e = rescale_exponent(warp_max(am));
            float s2 = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * 32 + lane < nvec) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float t = ldexpf(f[k], -e);
                        s2 = fmaf(t, t, s2);
                    }
                }
            rs = rstd_rescaled(warp_sum(s2), n_f, a.eps, e);
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V], wf[V], o[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = f[k] * rs * wf[k];
                st_stream(y4 + base + c, E::pack(o));
            }
        }
        if (lane == 0 && a.rstd) a.rstd[row] = rs;
    }
}

// Chunk c of row r = x (+ residual) as fp32: one 128-bit vector (VEC) or one element.
// Through L2 only (.cg), since the row is read again by the next pass.
template <typename T, bool VEC, bool FUSED>
__device__ __forceinline__ void load_r_chunk(const FwdArgs &a, int64_t base, int c,
                                             float (&f)[Elem<T>::kPerVec]) {
    using E = Elem<T>;
    if constexpr (VEC) {
        const int64_t vi = base / E::kPerVec + c;
        E::unpack(__ldcg(static_cast<const uint4 *>(a.x) + vi), f);
        if constexpr (FUSED) {
            float b[E::kPerVec];
            E::unpack(__ldcg(static_cast<const uint4 *>(a.res) + vi), b);
#pragma unroll
            for (int k = 0; k < E::kPerVec; ++k) f[k] += b[k];
        }
    } else {
        f[0] = E::load1(a.x, base + c);
        if constexpr (FUSED) f[0] += E::load1(a.res, base + c);
    }
}

// Two passes over each row; VEC selects 128-bit vectors (aligned rows) or single elements.
// Pass 2 recomputes r from x and residual (it never reads residual_out back), so the in-place
// forms residual_out == residual / x stay correct: each element is read by the thread that
// later writes it, before it writes it.
template <typename T, bool VEC, bool FUSED>
__global__ void __launch_bounds__(1024) fwd_stream(const FwdArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;
    __shared__ float slots[2][32];

    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);

    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * static_cast<int64_t>(a.N);
        float ss = 0.f;
        for (int c = tid; c < nchunk; c += nthr) {
            float f[W];
            load_r_chunk<T, VEC, FUSED>(a, base, c, f);
#pragma unroll
            for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
        }
        ss = cta_sum(ss, slots[parity]);
        parity ^= 1;
        float rs;
        if (!needs_rescale(ss)) {
            rs = rstd_plain(ss, n_f, a.eps);
        } else {  // rare: sum of squares out of fp32 range, or an all-zero row
            float am = 0.f;
            for (int c = tid; c < nchunk; c += nthr) {
                float f[W];
                load_r_chunk<T, VEC, FUSED>(a, base, c, f);
#pragma unroll
                for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(f[k]));
            }
            am = cta_max(am, slots[parity]);
            parity ^= 1;
            const int e = rescale_exponent(am);
            float s2 = 0.f;
            for (int c = tid; c < nchunk; c += nthr) {
                float f[W];
                load_r_chunk<T, VEC, FUSED>(a, base, c, f);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const float t = ldexpf(f[k], -e);
                    s2 = fmaf(t, t, s2);
                }
            }
            s2 = cta_sum(s2, slots[parity]);
            parity ^= 1;
            rs = rstd_rescaled(s2, n_f, a.eps, e);
        }
        for (int c = tid; c < nchunk; c += nthr) {
            if constexpr (VEC) {
                const int64_t vi = base / W + c;
                float f[W], wf[W], o[W];
                E::unpack(ld_stream(static_cast<const uint4 *>(a.x) + vi), f);
                if constexpr (FUSED) {
                    float b[W];
                    E::unpack(ld_stream(static_cast<const uint4 *>(a.res) + vi), b);
#pragma unroll
                    for (int k = 0; k < W; ++k) f[k] += b[k];
                    st_stream(static_cast<uint4 *>(a.res_out) + vi, E::pack(f));
                }
                E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
#pragma unroll
                for (int k = 0; k < W; ++k) o[k] = f[k] * rs * wf[k];
                st_stream(static_cast<uint4 *>(a.y) + vi, E::pack(o));
            } else {
                float f = E::load1(a.x, base + c);
                if constexpr (FUSED) {
                    f += E::load1(a.res, base + c);
                    E::store1(a.res_out, base + c, f);
                }
                E::store1(a.y, base + c, f * rs * E::load1(a.w, c));
            }
        }
        if (tid == 0 && a.rstd) a.rstd[row] = rs;
    }
}

// ----------------------------------------------------------------------------------------
// Host-side dispatch over the compiled instances.
// ----------------------------------------------------------------------------------------
template <typename T, bool FUSED>
const void *fwd_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&fwd_row_cta<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&fwd_row_cta<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&fwd_row_cta<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&fwd_row_cta<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_WARP:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&fwd_row_warp<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&fwd_row_warp<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&fwd_row_warp<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&fwd_row_warp<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&fwd_stream<T, true, FUSED>)
                         : reinterpret_cast<const void *>(&fwd_stream<T, false, FUSED>);
        case RRN_VARIANT_ROW_CLUSTER:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&fwd_row_cluster<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&fwd_row_cluster<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&fwd_row_cluster<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&fwd_row_cluster_v8<T, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_TMA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&fwd_row_tma<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&fwd_row_tma<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&fwd_row_tma<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&fwd_row_tma<T, 8, FUSED>);
                default: return nullptr;
            }
        default: return nullptr;
    }
}

template <typename T>
const void *fwd_kernel_ptr_any(bool fused, const Launch &l) {
    return fused ? fwd_kernel_ptr<T, true>(l) : fwd_kernel_ptr<T, false>(l);
}

template <typename T>
cudaError_t launch_fwd(const FwdArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = fwd_kernel_ptr_any<T>(a.res != nullptr, l);
    if (!k) return cudaErrorInvalidConfiguration;
    if (l.smem > 0) {
        cudaError_t e = allow_dynamic_smem(k, l.smem);
        if (e != cudaSuccess) return e;
    }
    FwdArgs args = a;
    args.stages = l.stages;
    void *params[] = {&args};
    const bool per_row = (l.variant == RRN_VARIANT_ROW_CTA || l.variant == RRN_VARIANT_ROW_WARP) && l.smem == 0;
    return enqueue(k, l, l.variant == RRN_VARIANT_ROW_CLUSTER ? l.cluster : 0, per_row, params, stream);
}

template <typename T>
int occupancy_fwd_t(bool fused, const Launch &l) {
    const void *k = fwd_kernel_ptr_any<T>(fused, l);
    if (!k) return 0;
    if (l.cluster > 0) return max_active_clusters(k, l);
    if (l.smem > 0 && allow_dynamic_smem(k, l.smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, l.threads, static_cast<size_t>(l.smem)) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rrn
