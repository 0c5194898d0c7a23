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
//   fwd_row_cta   one row per CTA, the row held in registers as 128-bit vectors; the grid
//                 walks rows with a grid-sized stride (persistent when the grid is smaller
//                 than M, one row per CTA when it is not). Used for N up to 16K (bf16).
//   fwd_row_warp  one row per warp, no barrier at all; for short rows (bf16 N <= 2048).
//   fwd_stream    one row per CTA in two passes over global memory (sum of squares, then
//                 normalise, re-reading the row from L2): any N and any alignment.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace rrn {

template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(fwd_max_threads(VPT))
    fwd_row_cta(const FwdArgs a) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    __shared__ float slots[2][32];

    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    const uint4 *r4 = static_cast<const uint4 *>(a.res);
    uint4 *ro4 = static_cast<uint4 *>(a.res_out);
    uint4 *y4 = static_cast<uint4 *>(a.y);
    const float n_f = static_cast<float>(a.N);

    // The weight row stays in registers for every row this CTA handles.
    uint4 wv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
    }

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
        float acc[VPT][V];
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                E::unpack(xv[v], acc[v]);
                if (FUSED) {
                    float b[V];
                    E::unpack(rv[v], b);
#pragma unroll
                    for (int k = 0; k < V; ++k) acc[v][k] += b[k];
                    st_stream(ro4 + base + c, E::pack(acc[v]));
                }
#pragma unroll
                for (int k = 0; k < V; ++k) ss = fmaf(acc[v][k], acc[v][k], ss);
            }
        }
        ss = cta_sum(ss, slots[parity]);
        parity ^= 1;
        float rs;
        if (!needs_rescale(ss)) {
            rs = rstd_plain(ss, n_f, a.eps);
        } else {  // rare: sum of squares out of fp32 range, or an all-zero row
            float am = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * nthr + tid < nvec)
#pragma unroll
                    for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(acc[v][k]));
            am = cta_max(am, slots[parity]);
            parity ^= 1;
            const int e = rescale_exponent(am);
            float s2 = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * nthr + tid < nvec)
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float t = ldexpf(acc[v][k], -e);
                        s2 = fmaf(t, t, s2);
                    }
            s2 = cta_sum(s2, slots[parity]);
            parity ^= 1;
            rs = rstd_rescaled(s2, n_f, a.eps, e);
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float wf[V], o[V];
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = acc[v][k] * rs * wf[k];
                st_stream(y4 + base + c, E::pack(o));
            }
        }
        if (tid == 0 && a.rstd) a.rstd[row] = rs;
    }
}

template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(256) fwd_row_warp(const FwdArgs a) {
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
        float acc[VPT][V];
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                E::unpack(xv[v], acc[v]);
                if (FUSED) {
                    float b[V];
                    E::unpack(rv[v], b);
#pragma unroll
                    for (int k = 0; k < V; ++k) acc[v][k] += b[k];
                    st_stream(ro4 + base + c, E::pack(acc[v]));
                }
#pragma unroll
                for (int k = 0; k < V; ++k) ss = fmaf(acc[v][k], acc[v][k], ss);
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
                if (v * 32 + lane < nvec)
#pragma unroll
                    for (int k = 0; k < V; ++k) am = fmaxf(am, fabsf(acc[v][k]));
            const int e = rescale_exponent(warp_max(am));
            float s2 = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * 32 + lane < nvec)
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float t = ldexpf(acc[v][k], -e);
                        s2 = fmaf(t, t, s2);
                    }
            rs = rstd_rescaled(warp_sum(s2), n_f, a.eps, e);
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float wf[V], o[V];
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = acc[v][k] * rs * wf[k];
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
    FwdArgs args = a;
    void *params[] = {&args};
    return cudaLaunchKernel(k, dim3(l.ctas), dim3(l.threads), params, 0, stream);
}

template <typename T>
int occupancy_fwd_t(bool fused, const Launch &l) {
    const void *k = fwd_kernel_ptr_any<T>(fused, l);
    if (!k) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, l.threads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rrn
