// Backward kernels of RMSNorm, with a two-stage deterministic dw.
//
// Per row (xhat = x * rstd, g = dy * w, c = sum(g * xhat) / N):
//   dx = rstd * (g - xhat * c)
// and dw = sum over rows of dy * xhat, reduced in two fixed-order stages:
//   stage 1  CTA p owns a contiguous block of rows; each thread keeps the dw partial sums of
//            its own columns in registers across those rows and writes them once to row p of
//            a [P, N] fp32 workspace.
//   stage 2  dw[j] = sum over p of workspace[p, j], in a fixed order (rows p = g, g+G, ...
//            per group g, then the G group sums in order). No atomics anywhere, so dw is
//            bitwise reproducible for a given (M, N, dtype, device).
// The pages give the op (Machete "Built-In Areas": RMSNorm and autograd helpers) but no
// backward formula; the one above is the exact derivative of the forward definition.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace rrn {

template <typename T, int VPT>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) bwd_row_cta(const BwdArgs a) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    __shared__ float slots[2][32];

    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const uint4 *dy4 = static_cast<const uint4 *>(a.dy);
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    uint4 *dx4 = static_cast<uint4 *>(a.dx);
    const float n_f = static_cast<float>(a.N);

    uint4 wv[VPT];
    float dw[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = 0.f;
    }

    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
    const int64_t row1 = min(a.M, row0 + a.rows_per_cta);
    int parity = 0;
    for (int64_t row = row0; row < row1; ++row) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], dyv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_stream(x4 + base + c);
                dyv[v] = ld_stream(dy4 + base + c);
            }
        }
        const float rs = __ldg(a.rstd + row);
        float xh[VPT][V], g[VPT][V];
        float dot = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float d[V], wf[V];
                E::unpack(xv[v], xh[v]);
                E::unpack(dyv[v], d);
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    xh[v][k] *= rs;
                    g[v][k] = d[k] * wf[k];
                    dot = fmaf(g[v][k], xh[v][k], dot);
                    dw[v][k] = fmaf(d[k], xh[v][k], dw[v][k]);
                }
            }
        }
        dot = cta_sum(dot, slots[parity]);
        parity ^= 1;
        const float cm = dot / n_f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float o[V];
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = rs * (g[v][k] - xh[v][k] * cm);
                st_stream(dx4 + base + c, E::pack(o));
            }
        }
    }

    float *prow = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float4 *dst = reinterpret_cast<float4 *>(prow + static_cast<int64_t>(c) * V);
#pragma unroll
            for (int q = 0; q < V / 4; ++q)
                dst[q] = make_float4(dw[v][4 * q], dw[v][4 * q + 1], dw[v][4 * q + 2], dw[v][4 * q + 3]);
        }
    }
}

// Two passes over each row (any N, any alignment); the dw partials live in the CTA's own
// workspace row instead of registers. Each workspace element is owned by one thread.
template <typename T, bool VEC>
__global__ void __launch_bounds__(1024) bwd_stream(const BwdArgs a) {
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;
    __shared__ float slots[2][32];

    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);
    float *prow = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;

    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
    const int64_t row1 = min(a.M, row0 + a.rows_per_cta);
    int parity = 0;
    for (int64_t row = row0; row < row1; ++row) {
        const int64_t base = row * static_cast<int64_t>(a.N);
        const float rs = __ldg(a.rstd + row);
        float dot = 0.f;
        for (int c = tid; c < nchunk; c += nthr) {
            float xf[W], df[W], wf[W];
            if constexpr (VEC) {
                const int64_t vi = base / W + c;
                E::unpack(__ldcg(static_cast<const uint4 *>(a.x) + vi), xf);
                E::unpack(__ldcg(static_cast<const uint4 *>(a.dy) + vi), df);
                E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
            } else {
                xf[0] = E::load1(a.x, base + c);
                df[0] = E::load1(a.dy, base + c);
                wf[0] = E::load1(a.w, c);
            }
#pragma unroll
            for (int k = 0; k < V; ++k) dot = fmaf(df[k] * wf[k], xf[k] * rs, dot);
        }
        dot = cta_sum(dot, slots[parity]);
        parity ^= 1;
        const float cm = dot / n_f;
        const bool first = (row == row0);
        for (int c = tid; c < nchunk; c += nthr) {
            float xf[W], df[W], wf[W], o[W];
            if constexpr (VEC) {
                const int64_t vi = base / W + c;
                E::unpack(ld_stream(static_cast<const uint4 *>(a.x) + vi), xf);
                E::unpack(ld_stream(static_cast<const uint4 *>(a.dy) + vi), df);
                E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
            } else {
                xf[0] = E::load1(a.x, base + c);
                df[0] = E::load1(a.dy, base + c);
                wf[0] = E::load1(a.w, c);
            }
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const float xh = xf[k] * rs;
                const float g = df[k] * wf[k];
                o[k] = rs * (g - xh * cm);
                float *pw = prow + static_cast<int64_t>(c) * V + k;
                *pw = first ? df[k] * xh : fmaf(df[k], xh, *pw);
            }
            if constexpr (VEC) {
                st_stream(static_cast<uint4 *>(a.dx) + base / W + c, E::pack(o));
            } else {
                E::store1(a.dx, base + c, o[0]);
            }
        }
    }
}

// Stage 2: dw[j] = sum_p partial[p, j]. A CTA covers 32 consecutive columns with
// kReduceThreads / 32 row groups; group g sums rows p = g, g + G, g + 2G, ... in order, then
// the first warp adds the G group sums in order.
__global__ void __launch_bounds__(kReduceThreads)
    bwd_dw_reduce(const float *__restrict__ partial, float *__restrict__ dw, int P, int N) {
    constexpr int G = kReduceThreads / 32;
    __shared__ float sums[G][32];
    const int lane = threadIdx.x & 31;
    const int grp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (col < N)
        for (int p = grp; p < P; p += G) acc += __ldcg(partial + static_cast<int64_t>(p) * N + col);
    sums[grp][lane] = acc;
    __syncthreads();
    if (grp == 0 && col < N) {
        float t = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) t += sums[g][lane];
        dw[col] = t;
    }
}

template <typename T>
const void *bwd_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&bwd_row_cta<T, 1>);
                case 2: return reinterpret_cast<const void *>(&bwd_row_cta<T, 2>);
                case 4: return reinterpret_cast<const void *>(&bwd_row_cta<T, 4>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&bwd_stream<T, true>)
                         : reinterpret_cast<const void *>(&bwd_stream<T, false>);
        default: return nullptr;
    }
}

// Stage 1 on l.ctas CTAs (each owning a.rows_per_cta rows), then stage 2, on one stream.
template <typename T>
cudaError_t launch_bwd(const BwdArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = bwd_kernel_ptr<T>(l);
    if (!k) return cudaErrorInvalidConfiguration;
    BwdArgs args = a;
    void *params[] = {&args};
    cudaError_t e = cudaLaunchKernel(k, dim3(l.ctas), dim3(l.threads), params, 0, stream);
    if (e != cudaSuccess) return e;
    const int blocks = (a.N + 31) / 32;
    bwd_dw_reduce<<<blocks, kReduceThreads, 0, stream>>>(a.partial, a.dw, l.ctas, a.N);
    return cudaGetLastError();
}

template <typename T>
int occupancy_bwd_t(const Launch &l) {
    const void *k = bwd_kernel_ptr<T>(l);
    if (!k) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, l.threads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rrn
