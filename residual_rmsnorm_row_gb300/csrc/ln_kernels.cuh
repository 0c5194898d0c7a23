// LayerNorm kernels: the mean-subtracting variant of the row norm, on the same skeleton as the
// RMSNorm kernels (the CuTe DSL skill page lists a "CTA norm (LayerNorm)" example in its
// "Workflow 0" example index; the kernels here are this library's own design).
//
// Forward, per row of r = x (+ residual) in fp32:
//   mean = sum(r) / N;  var = sum((r - mean)^2) / N;  rstd = rsqrt(var + eps)
//   (sums of deviations from a shift K near the mean, in one CTA-wide step, or the corrected
//   two-pass algorithm where K is far from the mean: never the cancellation-prone
//   sum(r^2) / N - mean^2; see ln_stats)
//   y = RN((r - mean) * rstd * w + b);  residual_out = RN(r);  mean, rstd stored as fp32
// Backward, with xhat = (x - mean) * rstd and g = dy * w:
//   dx = rstd * (g - mean(g) - xhat * mean(g * xhat))  (+ d_ro, fused)
//   dw = sum over rows of dy * xhat,  db = sum over rows of dy  (two fixed-order stages)
#pragma once

#include "bwd_kernels.cuh"
#include "common.cuh"
#include "launch.h"

namespace rrn {

// Sum of two floats over the CTA (one barrier); same fixed order as cta_sum.
__device__ __forceinline__ float2 cta_sum2(float a, float b, float (*slots)[32]) {
    a = warp_sum(a);
    b = warp_sum(b);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        slots[0][warp] = a;
        slots[1][warp] = b;
    }
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float2 t = make_float2(0.f, 0.f);
    for (int i = 0; i < nwarps; ++i) {
        t.x += slots[0][i];
        t.y += slots[1][i];
    }
    return t;
}

// ------------------------------------------------------------------------------ forward
// The row statistics from per-thread access to the row values: `each(fn)` calls fn(v) for
// every fp32 value of the row this thread owns. Returns (mean, rstd) as a reference value m0,
// a small correction corr (mean = m0 + corr) and rstd: deviations are formed as
// (r - m0) - corr, so the fp32 rounding of the mean itself never enters them. The reductions
// are those of `red` (CtaReduce or WarpReduce, below).
// ln_stats_two_pass: pass 1 gives a first mean m0 = sum(r) / N; pass 2 sums d = r - m0 and d^2
// together (one barrier) and corrects both: corr = sum(d) / N and
// sum((r - mean)^2) = sum(d^2) - sum(d)^2 / N (the corrected two-pass algorithm), so the
// rounding error of m0 - which grows with |mean|, not with the spread - cancels out.
// ln_stats (below) does the same in one step, relative to a shift from the row's first values,
// when that is safe.
struct LnStats {
    float m0;    // reference value: the first-pass mean or the shift of the one-step statistics
    float corr;  // mean - m0
    float rstd;
    __device__ __forceinline__ float mean() const { return m0 + corr; }
    __device__ __forceinline__ float dev(float r) const { return (r - m0) - corr; }
};

// The reductions the statistics take, over the CTA (two slot pairs in shared memory, used
// alternately, as cta_sum callers do) or over one warp (shuffles only, for a row per warp). Both
// add in a fixed order, so every thread of the group gets the same bits.
struct CtaReduce {
    float (&slots)[2][2][32];
    int &parity;
    __device__ __forceinline__ float sum(float v) {
        const float t = cta_sum(v, slots[parity][0]);
        parity ^= 1;
        return t;
    }
    __device__ __forceinline__ float max(float v) {
        const float t = cta_max(v, slots[parity][0]);
        parity ^= 1;
        return t;
    }
    __device__ __forceinline__ float2 sum2(float a, float b) {
        const float2 t = cta_sum2(a, b, slots[parity]);
        parity ^= 1;
        return t;
    }
};
__device__ __forceinline__ float2 red_warp_sum2(float a, float b) { return make_float2(warp_sum(a), warp_sum(b)); }
struct WarpReduce {
    __device__ __forceinline__ float sum(float v) const { return warp_sum(v); }
    __device__ __forceinline__ float max(float v) const { return warp_max(v); }
    __device__ __forceinline__ float2 sum2(float a, float b) const { return make_float2(warp_sum(a), warp_sum(b)); }
};

// The shift of the one-step statistics: the mean of the row's first min(N, 8) values r (formed
// as r_of forms them), which every thread computes from the same loads - the same bits
// everywhere - and which lies within a few sigma / sqrt(8) of the row mean in typical rows, so
// that the one-step statistics lose next to nothing to cancellation.
template <typename T, bool FUSED>
__device__ __forceinline__ float ln_shift(const void *x, const void *res, int64_t base, int N) {
    using E = Elem<T>;
    const int n = N < 8 ? N : 8;
    float s = 0.f;
    for (int k = 0; k < n; ++k) {
        float r = E::load1(x, base + k);
        if constexpr (FUSED) r += E::load1(res, base + k);
        s += r;
    }
    return s / static_cast<float>(n);
}

// ln_shift for the 128-bit vector kernels: the same values summed in the same order, read as
// the one or two vectors that hold them (vbase = the row's first vector).
template <typename T, bool FUSED>
__device__ __forceinline__ float ln_shift_vec(const void *x, const void *res, int64_t vbase, int N) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    const int n = N < 8 ? N : 8;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < (8 + V - 1) / V; ++c) {
        if (c * V >= n) break;
        const uint4 xv = __ldca(static_cast<const uint4 *>(x) + vbase + c);
        uint4 rv{};
        if constexpr (FUSED) rv = __ldca(static_cast<const uint4 *>(res) + vbase + c);
        float f[V];
        r_of<T, FUSED>(xv, rv, f);
#pragma unroll
        for (int k = 0; k < V; ++k)
            if (c * V + k < n) s += f[k];
    }
    return s / static_cast<float>(n);
}

// The corrected two-pass statistics (the fallback of ln_stats).
template <typename Red, typename Each>
__device__ __forceinline__ LnStats ln_stats_two_pass(Each each, float n_f, float eps, Red &red) {
    float s1 = 0.f;
    each([&](float v) { s1 += v; });
    s1 = red.sum(s1);
    float m0;
    if (isfinite(s1)) {
        m0 = s1 / n_f;
    } else {  // rare: the sum overflowed fp32 - add the row scaled by a power of two
        float am = 0.f;
        each([&](float v) { am = fmaxf(am, fabsf(v)); });
        am = red.max(am);
        const int e = rescale_exponent(am);
        float t = 0.f;
        each([&](float v) { t += ldexpf(v, -e); });
        t = red.sum(t);
        m0 = ldexpf(t / n_f, e);
    }
    float d1 = 0.f, d2 = 0.f;
    each([&](float v) {
        const float d = v - m0;
        d1 += d;
        d2 = fmaf(d, d, d2);
    });
    const float2 t2 = red.sum2(d1, d2);
    LnStats st;
    st.m0 = m0;
    st.corr = isfinite(t2.x) ? t2.x / n_f : 0.f;
    float rs;
    if (!needs_rescale(t2.y)) {
        const float ssd = fmaxf(t2.y - t2.x * (t2.x / n_f), 0.f);
        rs = rstd_plain(ssd, n_f, eps);
    } else {  // rare: squared deviations out of fp32 range, or a constant row
        float am = 0.f;
        each([&](float v) { am = fmaxf(am, fabsf(st.dev(v))); });
        am = red.max(am);
        const int e = rescale_exponent(am);
        float t = 0.f;
        each([&](float v) {
            const float d = ldexpf(st.dev(v), -e);
            t = fmaf(d, d, t);
        });
        t = red.sum(t);
        rs = rstd_rescaled(t, n_f, eps, e);
    }
    st.rstd = rs;
    return st;
}

// One CTA-wide step in the common case: with K the mean of the row's first values (ln_shift),
// sum d = r - K and d^2 together; then mean = K + sum(d) / N and
// sum((r - mean)^2) = sum(d^2) - sum(d)^2 / N. The subtraction loses precision only when K sits
// far from the mean compared with the spread: the result is kept when
// sum((r - mean)^2) >= sum(d^2) / 16 (at most four bits of cancellation - and in typical rows
// well under one, as K is within about sigma / sqrt(8) of the mean) and the sums are in range;
// otherwise - a constant row, outliers among the first values, overflow - the row gets the
// corrected two-pass statistics (ln_stats_two_pass). As there, m0 (= K) and the correction stay
// apart.
// ln_stats_shifted takes this thread's sums d1 = sum(r - K), d2 = sum((r - K)^2), which a kernel
// may have formed in a pass of its own (the row-per-CTA forward forms them while it stores
// residual_out); ln_stats forms them itself.
template <typename Red, typename Each>
__device__ __forceinline__ LnStats ln_stats_shifted(Each each, float K, float d1, float d2, float n_f,
                                                    float eps, Red &red) {
    const float2 t = red.sum2(d1, d2);
    if (isfinite(t.x) && !needs_rescale(t.y)) {
        const float corr = t.x / n_f;
        const float ssd = t.y - t.x * corr;
        if (ssd >= 0.0625f * t.y) {
            LnStats st;
            st.m0 = K;
            st.corr = corr;
            st.rstd = rstd_plain(ssd, n_f, eps);
            return st;
        }
    }
    return ln_stats_two_pass(each, n_f, eps, red);
}

template <typename Red, typename Each>
__device__ __forceinline__ LnStats ln_stats(Each each, float K, float n_f, float eps, Red &red) {
    float d1 = 0.f, d2 = 0.f;
    each([&](float v) {
        const float d = v - K;
        d1 += d;
        d2 = fmaf(d, d, d2);
    });
    return ln_stats_shifted(each, K, d1, d2, n_f, eps, red);
}

// The forward's per-vector arithmetic, in packed fp32 pairs (PACKED) or one value at a time;
// both give the same values, except that the pairs keep two partial sums where one value at a
// time keeps one. Packed pairs issue half the floating-point instructions but hold more
// registers: the row-per-CTA forward uses them from 4 vectors per thread up, where its register
// cap leaves room (at 2 they made it spill).
// r = x (+ residual):
template <typename T, bool FUSED, bool PACKED>
__device__ __forceinline__ void ln_r_of(const uint4 &xv, const uint4 &rv, float (&f)[Elem<T>::kPerVec]) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    if constexpr (!PACKED) {
        r_of<T, FUSED>(xv, rv, f);
    } else {
        E::unpack(xv, f);
        if constexpr (FUSED) {
            float rf[V];
            E::unpack(rv, rf);
#pragma unroll
            for (int k = 0; k < V; k += 2) {
                const float2 t = add2(pair(f[k], f[k + 1]), pair(rf[k], rf[k + 1]));
                f[k] = t.x;
                f[k + 1] = t.y;
            }
        }
    }
}

// d1 += sum(r - K), d2 += sum((r - K)^2) over the vector (one value at a time: in d1.x, d2.x):
template <int V, bool PACKED>
__device__ __forceinline__ void ln_moments(const float (&f)[V], float K, float2 &d1, float2 &d2) {
#pragma unroll
    for (int k = 0; k < V; k += PACKED ? 2 : 1) {
        if constexpr (PACKED) {
            const float2 d = add2(pair(f[k], f[k + 1]), splat(-K));
            d1 = add2(d1, d);
            d2 = fma2(d, d, d2);
        } else {
            const float d = f[k] - K;
            d1.x += d;
            d2.x = fmaf(d, d, d2.x);
        }
    }
}

// y = ((r - m0) * rstd + ncr) * w + b, where ncr = -corr * rstd:
template <int V, bool PACKED>
__device__ __forceinline__ void ln_out(const float (&f)[V], const float (&wf)[V], const float (&bf)[V],
                                       float m0, float rstd, float ncr, float (&o)[V]) {
#pragma unroll
    for (int k = 0; k < V; k += PACKED ? 2 : 1) {
        if constexpr (PACKED) {
            const float2 t = fma2(add2(pair(f[k], f[k + 1]), splat(-m0)), splat(rstd), splat(ncr));
            const float2 u = fma2(t, pair(wf[k], wf[k + 1]), pair(bf[k], bf[k + 1]));
            o[k] = u.x;
            o[k + 1] = u.y;
        } else {
            o[k] = fmaf(fmaf(f[k] - m0, rstd, ncr), wf[k], bf[k]);
        }
    }
}

// Row per CTA (rows in registers). w and b are read where they are used, from L1 (prefetched
// there at the start), rather than held in registers: with the register cap that keeps more
// CTAs - more rows in flight - per SM, as in the RMSNorm forward.
template <typename T, int VPT, bool FUSED>
__global__ void __maxnreg__(fwd_max_regs(VPT)) ln_fwd_row_cta(const LnFwdArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    constexpr bool P = VPT >= 4;  // packed fp32 pairs
    __shared__ float slots[2][2][32];
    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);
    const uint4 *w4 = static_cast<const uint4 *>(a.w);
    const uint4 *b4 = static_cast<const uint4 *>(a.b);

#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            prefetch_l1(w4 + c);
            if (b4) prefetch_l1(b4 + c);
        }
    }
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                if (FUSED) rv[v] = ld_stream(static_cast<const uint4 *>(a.res) + base + c);
            }
        }
        const float K = ln_shift_vec<T, FUSED>(a.x, a.res, base, a.N);
        // residual_out is stored in the same pass, except the vectors that hold the values K is
        // formed from: residual_out may be the buffer of x or residual, and other warps may not
        // have read them yet; those are stored after the CTA-wide sums (a barrier) below
        float2 d1 = splat(0.f), d2 = splat(0.f);  // sums of d = r - K and d^2
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float f[V];
                ln_r_of<T, FUSED, P>(xv[v], rv[v], f);
                if (FUSED && c * V >= 8) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                ln_moments<V, P>(f, K, d1, d2);
            }
        }
        auto each = [&](auto fn) {
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * nthr + tid < nvec) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) fn(f[k]);
                }
        };
        CtaReduce red{slots, parity};
        const LnStats st = ln_stats_shifted(each, K, d1.x + d1.y, d2.x + d2.y, n_f, a.eps, red);
        const float ncr = -st.corr * st.rstd;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float f[V], wf[V], bf[V], o[V];
                ln_r_of<T, FUSED, P>(xv[v], rv[v], f);
                E::unpack(ld_keep(w4 + c), wf);
                if (b4) {
                    E::unpack(ld_keep(b4 + c), bf);
                } else {
#pragma unroll
                    for (int k = 0; k < V; ++k) bf[k] = 0.f;
                }
                // (r - m0 - corr) * rstd with one operation fewer: (r - m0) * rstd - corr * rstd
                ln_out<V, P>(f, wf, bf, st.m0, st.rstd, ncr, o);
                if (FUSED && c * V < 8) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                st_stream(static_cast<uint4 *>(a.y) + base + c, E::pack(o));
            }
        }
        if (tid == 0) {
            if (a.mean) a.mean[row] = st.mean();
            if (a.rstd) a.rstd[row] = st.rstd;
        }
    }
}

// Row per warp, for short rows over many rows (as the RMSNorm forward's fwd_row_warp): lane l
// owns vectors v * 32 + l, the statistics are warp-wide (shuffles, no barrier), and warps walk
// rows with a grid-sized stride. Nothing but the row's own loads stands before its arithmetic:
// w and b are loaded into registers once, and the shift K (the mean of the row's first 8
// values, added up per vector and then over the lanes that hold them) is passed round by
// shuffles from the lanes that loaded those values.
template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(256) ln_fwd_row_warp(const LnFwdArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    constexpr int KL = (8 + V - 1) / V;  // lanes whose vector 0 holds the row's first 8 values
    constexpr bool P = VPT >= 4;  // packed fp32 pairs
    const int nvec = a.N / V;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const float n_f = static_cast<float>(a.N);
    const int nk = a.N < 8 ? a.N : 8;
    const float inv_nk = 1.f / static_cast<float>(nk);
    uint4 wv[VPT], bv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * 32 + lane;
        if (c < nvec) {
            wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
            bv[v] = a.b ? ld_keep(static_cast<const uint4 *>(a.b) + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    WarpReduce red;
    for (int64_t row = warp0; row < a.M; row += nwarps) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                if (FUSED) rv[v] = ld_stream(static_cast<const uint4 *>(a.res) + base + c);
            }
        }
        float ks = 0.f;
        if (lane < KL && lane < nvec) {
            float f[V];
            r_of<T, FUSED>(xv[0], rv[0], f);
#pragma unroll
            for (int k = 0; k < V; ++k)
                if (lane * V + k < nk) ks += f[k];
        }
        float K = __shfl_sync(0xffffffffu, ks, 0);
#pragma unroll
        for (int l = 1; l < KL; ++l) K += __shfl_sync(0xffffffffu, ks, l);
        K *= inv_nk;
        // (residual_out may be the buffer of x or residual: each lane stores only the vectors it
        // has itself loaded, and the values K is formed from travelled by shuffle)
        float2 d1 = splat(0.f), d2 = splat(0.f);  // sums of d = r - K and d^2
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V];
                ln_r_of<T, FUSED, P>(xv[v], rv[v], f);
                if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                ln_moments<V, P>(f, K, d1, d2);
            }
        }
        auto each = [&](auto fn) {
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (v * 32 + lane < nvec) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) fn(f[k]);
                }
        };
        const LnStats st = ln_stats_shifted(each, K, d1.x + d1.y, d2.x + d2.y, n_f, a.eps, red);
        const float ncr = -st.corr * st.rstd;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V], wf[V], bf[V], o[V];
                ln_r_of<T, FUSED, P>(xv[v], rv[v], f);
                E::unpack(opaque(wv[v]), wf);
                E::unpack(opaque(bv[v]), bf);
                ln_out<V, P>(f, wf, bf, st.m0, st.rstd, ncr, o);
                st_stream(static_cast<uint4 *>(a.y) + base + c, E::pack(o));
            }
        }
        if (lane == 0) {
            if (a.mean) a.mean[row] = st.mean();
            if (a.rstd) a.rstd[row] = st.rstd;
        }
    }
}

// Any N, any alignment: every pass re-reads the row (from L2); VEC selects 128-bit vectors.
template <typename T, bool VEC, bool FUSED>
__global__ void __launch_bounds__(1024) ln_fwd_stream(const LnFwdArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;
    __shared__ float slots[2][2][32];
    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);

    auto load_r = [&](int64_t base, int c, float (&f)[W]) {
        if constexpr (VEC) {
            const int64_t vi = base / W + c;
            E::unpack(__ldcg(static_cast<const uint4 *>(a.x) + vi), f);
            if constexpr (FUSED) {
                float bb[W];
                E::unpack(__ldcg(static_cast<const uint4 *>(a.res) + vi), bb);
#pragma unroll
                for (int k = 0; k < W; ++k) f[k] += bb[k];
            }
        } else {
            f[0] = E::load1(a.x, base + c);
            if constexpr (FUSED) f[0] += E::load1(a.res, base + c);
        }
    };
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * static_cast<int64_t>(a.N);
        auto each = [&](auto fn) {
            for (int c = tid; c < nchunk; c += nthr) {
                float f[W];
                load_r(base, c, f);
#pragma unroll
                for (int k = 0; k < V; ++k) fn(f[k]);
            }
        };
        const float K = ln_shift<T, FUSED>(a.x, a.res, base, a.N);
        CtaReduce red{slots, parity};
        const LnStats st = ln_stats(each, K, n_f, a.eps, red);
        for (int c = tid; c < nchunk; c += nthr) {
            float f[W], wf[W], bf[W], o[W];
            load_r(base, c, f);
            if constexpr (VEC) {
                E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
                if (a.b) E::unpack(ld_keep(static_cast<const uint4 *>(a.b) + c), bf);
            } else {
                wf[0] = E::load1(a.w, c);
                if (a.b) bf[0] = E::load1(a.b, c);
            }
            if (!a.b)
#pragma unroll
                for (int k = 0; k < V; ++k) bf[k] = 0.f;
#pragma unroll
            for (int k = 0; k < V; ++k) o[k] = fmaf(st.dev(f[k]) * st.rstd, wf[k], bf[k]);
            if constexpr (VEC) {
                if constexpr (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base / W + c, E::pack(f));
                st_stream(static_cast<uint4 *>(a.y) + base / W + c, E::pack(o));
            } else {
                if constexpr (FUSED) E::store1(a.res_out, base + c, f[0]);
                E::store1(a.y, base + c, o[0]);
            }
        }
        if (tid == 0) {
            if (a.mean) a.mean[row] = st.mean();
            if (a.rstd) a.rstd[row] = st.rstd;
        }
    }
}

// ------------------------------------------------------------------------------ backward
// One vector (V values, V even) of a row in the backward, in packed fp32 pairs: with
// xhat = (x - mean) * rstd and g = dy * w, adds dy * xhat into dw, dy into db, and g and
// g * xhat into the row's two running sums (kept as pairs, added up once per row).
template <int V>
__device__ __forceinline__ void ln_bwd_accumulate(const float (&xf)[V], const float (&d)[V],
                                                  const float (&wf)[V], float mu, float rs,
                                                  float (&dw)[V], float (&db)[V], float2 &sg,
                                                  float2 &sgx) {
#pragma unroll
    for (int k = 0; k < V; k += 2) {
        const float2 d2 = pair(d[k], d[k + 1]);
        const float2 xh = mul2(add2(pair(xf[k], xf[k + 1]), splat(-mu)), splat(rs));
        const float2 g = mul2(d2, pair(wf[k], wf[k + 1]));
        sg = add2(sg, g);
        sgx = fma2(g, xh, sgx);
        const float2 w2 = fma2(d2, xh, pair(dw[k], dw[k + 1]));
        const float2 b2 = add2(pair(db[k], db[k + 1]), d2);
        dw[k] = w2.x;
        dw[k + 1] = w2.y;
        db[k] = b2.x;
        db[k + 1] = b2.y;
    }
}

// dx for one vector: rstd * (g - mean(g) - xhat * mean(g * xhat)), evaluated as
// g * rstd + (xhat * cx + c) with cx = -rstd * mean(g * xhat), c = -rstd * mean(g).
template <int V>
__device__ __forceinline__ void ln_bwd_dx(const float (&xf)[V], const float (&d)[V],
                                          const float (&wf)[V], float mu, float rs, float cx,
                                          float c, float (&o)[V]) {
#pragma unroll
    for (int k = 0; k < V; k += 2) {
        const float2 xh = mul2(add2(pair(xf[k], xf[k + 1]), splat(-mu)), splat(rs));
        const float2 g = mul2(pair(d[k], d[k + 1]), pair(wf[k], wf[k + 1]));
        const float2 r = fma2(g, splat(rs), fma2(xh, splat(cx), splat(c)));
        o[k] = r.x;
        o[k + 1] = r.y;
    }
}

// One row of the backward with its x, dy (and d_ro) vectors in registers (this thread owns
// vectors c = v * blockDim.x + threadIdx.x; mu, rs the row's mean and rstd): dx written, and
// dy * xhat and dy added into this thread's dw and db registers. w is read where it is used,
// from L1, rather than held in registers: this kernel's registers go to the dw and db sums.
template <typename T, int VPT, bool ADDG>
__device__ __forceinline__ void ln_bwd_row_body(const LnBwdArgs &a, int64_t row, int nvec,
                                                const uint4 (&xv)[VPT], const uint4 (&dyv)[VPT],
                                                const uint4 (&gv)[VPT],
                                                float (&dw)[VPT][Elem<T>::kPerVec],
                                                float (&db)[VPT][Elem<T>::kPerVec],
                                                float (&slots)[2][2][32], int &parity, float mu,
                                                float rs) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);
    const uint4 *w4 = static_cast<const uint4 *>(a.w);
    float2 sg = splat(0.f), sgx = splat(0.f);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float xf[V], d[V], wf[V];
            E::unpack(xv[v], xf);
            E::unpack(dyv[v], d);
            E::unpack(ld_keep(w4 + c), wf);
            ln_bwd_accumulate<V>(xf, d, wf, mu, rs, dw[v], db[v], sg, sgx);
        }
    }
    const float2 t = cta_sum2(sg.x + sg.y, sgx.x + sgx.y, slots[parity]);
    parity ^= 1;
    const float cx = -rs * (t.y * inv_n), cc = -rs * (t.x * inv_n);
    const int64_t base = row * nvec;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float xf[V], d[V], wf[V], o[V];
            E::unpack(xv[v], xf);
            E::unpack(dyv[v], d);
            E::unpack(ld_keep(w4 + c), wf);
            ln_bwd_dx<V>(xf, d, wf, mu, rs, cx, cc, o);
            if constexpr (ADDG) {
                float gg[V];
                E::unpack(gv[v], gg);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] += gg[k];
            }
            st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
        }
    }
}

// Stage 1 for short rows: a row per warp (as the RMSNorm backward's bwd_row_warp). Warp w of CTA
// p takes rows p * W + w, then every (P * W)-th row; lane l owns vectors v * 32 + l; the row's
// two sums are warp-wide (no barrier per row); dw and db stay in registers, and at the end the
// W warps' sums are added in warp order through shared memory (2 N floats) into rows p of the
// two workspace halves. (Loading the next row before the current row's arithmetic measured
// slower, as in bwd_row_warp: 131072 x 512 bf16 89.8 against 80.9 us.)
template <typename T, int VPT, bool ADDG>
__global__ void __launch_bounds__(256) ln_bwd_row_warp(const LnBwdArgs a) {
    pdl_enter();  // the stage-2 reduction may be scheduled from now on
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    extern __shared__ __align__(16) float red[];  // [2][N]: dw, then db
    const int nvec = a.N / V;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * W;
    const float inv_n = 1.f / static_cast<float>(a.N);
    const uint4 *dy4 = static_cast<const uint4 *>(a.dy);
    const uint4 *g4 = static_cast<const uint4 *>(a.d_ro);
    const uint4 *x4 = static_cast<const uint4 *>(a.x);

    uint4 wv[VPT];
    float dw[VPT][V], db[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * 32 + lane;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = db[v][k] = 0.f;
    }
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * W + warp; row < a.M; row += nw) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], dyv[VPT], gv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                xv[v] = ld_stream(x4 + base + c);
                dyv[v] = ld_stream(dy4 + base + c);
                if constexpr (ADDG) gv[v] = ld_stream(g4 + base + c);
            }
        }
        const float mu = __ldg(a.mean + row);
        const float rs = __ldg(a.rstd + row);
        float2 sg = splat(0.f), sgx = splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float xf[V], d[V], wf[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(opaque(wv[v]), wf);
                ln_bwd_accumulate<V>(xf, d, wf, mu, rs, dw[v], db[v], sg, sgx);
            }
        }
        const float2 t = red_warp_sum2(sg.x + sg.y, sgx.x + sgx.y);
        const float cx = -rs * (t.y * inv_n), cc = -rs * (t.x * inv_n);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float xf[V], d[V], wf[V], o[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(opaque(wv[v]), wf);
                ln_bwd_dx<V>(xf, d, wf, mu, rs, cx, cc, o);
                if constexpr (ADDG) {
                    float gg[V];
                    E::unpack(gv[v], gg);
#pragma unroll
                    for (int k = 0; k < V; ++k) o[k] += gg[k];
                }
                st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
            }
        }
    }
    // the W warps' sums, added in warp order, then rows blockIdx.x of the workspace halves
    float *rw = red, *rb = red + a.N;
    for (int w = 0; w < W; ++w) {
        if (warp == w) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = v * 32 + lane;
                if (c < nvec) {
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        rw[c * V + k] = w == 0 ? dw[v][k] : rw[c * V + k] + dw[v][k];
                        rb[c * V + k] = w == 0 ? db[v][k] : rb[c * V + k] + db[v][k];
                    }
                }
            }
        }
        __syncthreads();
    }
    float *pw = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
    float *pb = a.partial + (static_cast<int64_t>(gridDim.x) + blockIdx.x) * a.N;
    for (int j = threadIdx.x; j < a.N; j += blockDim.x) {
        pw[j] = rw[j];
        pb[j] = rb[j];
    }
}

// This CTA's dw and db partial sums -> row blockIdx.x of the two [P, N] workspace halves.
template <typename T, int VPT>
__device__ __forceinline__ void ln_bwd_store_partial(const LnBwdArgs &a, int nvec,
                                                     const float (&dw)[VPT][Elem<T>::kPerVec],
                                                     const float (&db)[VPT][Elem<T>::kPerVec]) {
    constexpr int V = Elem<T>::kPerVec;
    float *pw = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
    float *pb = a.partial + (static_cast<int64_t>(gridDim.x) + blockIdx.x) * a.N;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * blockDim.x + threadIdx.x;
        if (c < nvec) {
#pragma unroll
            for (int q = 0; q < V / 4; ++q) {
                reinterpret_cast<float4 *>(pw + static_cast<int64_t>(c) * V)[q] =
                    make_float4(dw[v][4 * q], dw[v][4 * q + 1], dw[v][4 * q + 2], dw[v][4 * q + 3]);
                reinterpret_cast<float4 *>(pb + static_cast<int64_t>(c) * V)[q] =
                    make_float4(db[v][4 * q], db[v][4 * q + 1], db[v][4 * q + 2], db[v][4 * q + 3]);
            }
        }
    }
}

// Stage 1, rows in registers: CTA p owns rows p, p + P, p + 2P, ...; dw and db partials stay in
// registers and go to rows p of the two [P, N] workspace halves.
template <typename T, int VPT, bool ADDG>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) ln_bwd_row_cta(const LnBwdArgs a) {
    pdl_enter();  // the stage-2 reduction may be scheduled from now on
    constexpr int V = Elem<T>::kPerVec;
    __shared__ float slots[2][2][32];
    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;

    float dw[VPT][V], db[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) prefetch_l1(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = db[v][k] = 0.f;
    }
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], dyv[VPT], gv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                dyv[v] = ld_stream(static_cast<const uint4 *>(a.dy) + base + c);
                if constexpr (ADDG) gv[v] = ld_stream(static_cast<const uint4 *>(a.d_ro) + base + c);
            }
        }
        ln_bwd_row_body<T, VPT, ADDG>(a, row, nvec, xv, dyv, gv, dw, db, slots, parity,
                                      __ldg(a.mean + row), __ldg(a.rstd + row));
    }
    ln_bwd_store_partial<T, VPT>(a, nvec, dw, db);
}

// Stage 1 fed by the TMA engine: CTA p owns rows p, p + P, ..., keeps a.stages (>= 2) of them
// (x, dy and, fused, d_ro) in a shared-memory ring filled with cp.async.bulk, and reads each row
// from the ring twice - for the sums, and again for dx - instead of holding it in registers
// across the CTA-wide sums (the dw and db sums already take most of the registers: without the
// row, 2 vectors a thread fit in 80 registers, 3 CTAs of 256 threads per SM). So a slot is free
// only after the row's second pass: slot k % S is refilled (with row k - 1 + S) at the barrier
// of row k + 1, which every thread reaches after row k's second pass, and S - 1 rows are in
// flight while a row is worked on. The next row's mean and rstd are requested one row ahead.
constexpr int ln_bwd_ring_max_regs(int vpt) { return vpt == 2 ? 80 : vpt >= 4 ? 255 : 128; }
template <typename T, int VPT, bool ADDG>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) __maxnreg__(ln_bwd_ring_max_regs(VPT))
    ln_bwd_row_tma(const LnBwdArgs a) {
    pdl_enter();  // the stage-2 reduction may be scheduled from now on
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    constexpr int NT = ADDG ? 3 : 2;
    extern __shared__ __align__(128) unsigned char ring_buf[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ float slots[2][2][32];
    __shared__ int abort_flag;

    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);  // the row means below: one product each
    const uint4 *w4 = static_cast<const uint4 *>(a.w);
    RowRing<NT> ring;
    ring.buf = ring_buf;
    ring.full = full;
    ring.src[0] = static_cast<const char *>(a.x);
    ring.src[1] = static_cast<const char *>(a.dy);
    if constexpr (ADDG) ring.src[NT - 1] = static_cast<const char *>(a.d_ro);
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

    float dw[VPT][V], db[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) prefetch_l1(w4 + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = db[v][k] = 0.f;
    }
    auto vec = [&](int t, int c) {  // vector c of tensor t of the row under the ring's cursor
        return ld_shared_v4(ring.slot(t) + static_cast<size_t>(c) * 16);
    };
    int parity = 0;
    int64_t k = 0;
    float mu = 0.f, rs = 0.f;
    if (ring.nrows > 0) {
        mu = __ldg(a.mean + ring.first);
        rs = __ldg(a.rstd + ring.first);
    }
    for (; k < ring.nrows; ++k) {
        float mu_next = 0.f, rs_next = 0.f;
        if (k + 1 < ring.nrows) {
            const int64_t nxt = ring.first + (k + 1) * ring.stride;
            mu_next = __ldg(a.mean + nxt);
            rs_next = __ldg(a.rstd + nxt);
        }
        if (!ring.wait(a.faults)) abort_flag = 1;
        float2 sg = splat(0.f), sgx = splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float xf[V], d[V], wf[V];
                E::unpack(vec(0, c), xf);
                E::unpack(vec(1, c), d);
                E::unpack(ld_keep(w4 + c), wf);
                ln_bwd_accumulate<V>(xf, d, wf, mu, rs, dw[v], db[v], sg, sgx);
            }
        }
        // past this barrier every thread is done with row k's first pass and row k - 1's second
        const float2 t = cta_sum2(sg.x + sg.y, sgx.x + sgx.y, slots[parity]);
        parity ^= 1;
        if (abort_flag) break;  // written before the barrier: uniform
        if (tid == 0 && k >= 1 && k - 1 + ring.S < ring.nrows) {
            fence_proxy_async();
            ring.issue(k - 1 + ring.S, ring.prev());
        }
        // and the row after the ring's reach asked into L2, so that its bulk copy finds it there
        // (16384 x 4096 plain: 90.8 -> 86.5 us; 8192 x 8192: 97.1 -> 90.9 plain, 113.3 -> 105.5
        // fused; 16384 x 4096 fused: 102.6 -> 103.6)
        if (tid == 0 && k + ring.S < ring.nrows) {
            const int64_t off = (ring.first + (k + ring.S) * ring.stride) * static_cast<int64_t>(ring.row_bytes);
#pragma unroll
            for (int t = 0; t < NT; ++t) prefetch_l2_bulk(ring.src[t] + off, ring.row_bytes);
        }
        const float cx = -rs * (t.y * inv_n), cc = -rs * (t.x * inv_n);
        const int64_t base = (ring.first + k * ring.stride) * nvec;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float xf[V], d[V], wf[V], o[V];
                E::unpack(vec(0, c), xf);
                E::unpack(vec(1, c), d);
                E::unpack(ld_keep(w4 + c), wf);
                ln_bwd_dx<V>(xf, d, wf, mu, rs, cx, cc, o);
                if constexpr (ADDG) {
                    float gg[V];
                    E::unpack(vec(NT - 1, c), gg);
#pragma unroll
                    for (int j = 0; j < V; ++j) o[j] += gg[j];
                }
                st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
            }
        }
        ring.advance();
        mu = mu_next;
        rs = rs_next;
    }
    if (k < ring.nrows) {  // a wait ran out: the partial rows are not written; the fault word tells
        if (tid == 0) ring.drain(k, ring.S - 1);  // rows k .. k + S - 2 are in flight
        return;
    }
    ln_bwd_store_partial<T, VPT>(a, nvec, dw, db);
}

// Stage 1 for rows too wide for one CTA's dw and db registers, each row split across the C CTAs
// of a thread-block cluster (as the RMSNorm backward's bwd_row_split): CTA rank q owns the
// vectors [q * chunk, (q + 1) * chunk) of every row its cluster handles and keeps the dw and db
// partial sums of those columns; the row's two sums (of g and of g * xhat) are the sums of the C
// CTAs' parts, exchanged through distributed shared memory (ClusterExchange: asynchronous remote
// stores counted on mbarriers, no cluster barrier per row; every CTA adds the C pairs in rank
// order). Cluster k owns
// rows k, k + K, ... (K clusters) and writes its dw sums to row k and its db sums to row K + k
// of the workspace.
template <typename T, int VPT, bool ADDG>
__device__ __forceinline__ void ln_bwd_row_split_body(const LnBwdArgs &a) {
    pdl_enter();  // the stage-2 reduction may be scheduled from now on
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    __shared__ float slots[2][2][32];
    __shared__ float2 part[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    ClusterExchange<float2, kMaxCluster> xchg(part, xbar);

    const int nvec = a.N / V;
    const int C = static_cast<int>(cluster_nctarank());
    const int q = static_cast<int>(cluster_ctarank());
    const int chunk = (nvec + C - 1) / C;
    const int c0 = min(nvec, q * chunk);
    const int c1 = min(nvec, c0 + chunk);
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);
    const uint4 *w4 = static_cast<const uint4 *>(a.w);
    if (tid == 0) xchg.init();
    cluster_sync();  // every CTA of the cluster runs and has its barriers initialised

    float dw[VPT][V], db[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) prefetch_l1(w4 + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = db[v][k] = 0.f;
    }
    int parity = 0;
    const int64_t first = cluster_id_x();
    const int64_t ncl = cluster_nclusters_x();
    for (int64_t row = first; row < a.M; row += ncl) {
        const float mu = __ldg(a.mean + row);
        const float rs = __ldg(a.rstd + row);
        const int64_t base = row * nvec;
        {
            // ask L2 for this CTA's slices of the cluster's next row now, so that its loads find
            // them there (8192 x 16384 bf16 with the gradient at residual_out: 347 -> 297 us behind
            // a cluster barrier per row)
            const int64_t nxt = row + ncl;
            if (tid == 0 && c1 > c0 && nxt < a.M) {
                const int64_t nb = nxt * nvec + c0;
                const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
                prefetch_l2_bulk(static_cast<const uint4 *>(a.x) + nb, bytes);
                prefetch_l2_bulk(static_cast<const uint4 *>(a.dy) + nb, bytes);
                if constexpr (ADDG) prefetch_l2_bulk(static_cast<const uint4 *>(a.d_ro) + nb, bytes);
            }
        }
        uint4 xv[VPT], dyv[VPT], gv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                dyv[v] = ld_stream(static_cast<const uint4 *>(a.dy) + base + c);
                if constexpr (ADDG) gv[v] = ld_stream(static_cast<const uint4 *>(a.d_ro) + base + c);
            }
        }
        float2 sg = splat(0.f), sgx = splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float xf[V], d[V], wf[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(ld_keep(w4 + c), wf);
                ln_bwd_accumulate<V>(xf, d, wf, mu, rs, dw[v], db[v], sg, sgx);
            }
        }
        const float2 t = cta_sum2(sg.x + sg.y, sgx.x + sgx.y, slots[parity]);
        parity ^= 1;
        const float2 tt = xchg(t, make_float2(0.f, 0.f),
                               [](float2 u, float2 v) { return make_float2(u.x + v.x, u.y + v.y); },
                               a.faults);
        const float cx = -rs * (tt.y * inv_n), cc = -rs * (tt.x * inv_n);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float xf[V], d[V], wf[V], o[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(ld_keep(w4 + c), wf);
                ln_bwd_dx<V>(xf, d, wf, mu, rs, cx, cc, o);
                if constexpr (ADDG) {
                    float gg[V];
                    E::unpack(gv[v], gg);
#pragma unroll
                    for (int k = 0; k < V; ++k) o[k] += gg[k];
                }
                st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
            }
        }
    }
    float *pw = a.partial + first * a.N;
    float *pb = a.partial + (ncl + first) * a.N;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) {
#pragma unroll
            for (int i = 0; i < V / 4; ++i) {
                reinterpret_cast<float4 *>(pw + static_cast<int64_t>(c) * V)[i] =
                    make_float4(dw[v][4 * i], dw[v][4 * i + 1], dw[v][4 * i + 2], dw[v][4 * i + 3]);
                reinterpret_cast<float4 *>(pb + static_cast<int64_t>(c) * V)[i] =
                    make_float4(db[v][4 * i], db[v][4 * i + 1], db[v][4 * i + 2], db[v][4 * i + 3]);
            }
        }
    }
    cluster_sync();  // no CTA leaves while a peer's remote stores may still be on their way to it
}

// The split-row kernel; with the gradient at residual_out at 2 vectors a thread capped at 80
// registers (96 otherwise, no spills: 6 CTAs of 128 threads per SM instead of 5; bf16 8192 x
// 16384 190.8 -> 186.8 us, 4096 x 32768 215.4 -> 205.1 us). The other forms keep the compiler's
// own allocation.
template <typename T, int VPT, bool ADDG>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) ln_bwd_row_split(const LnBwdArgs a) {
    ln_bwd_row_split_body<T, VPT, ADDG>(a);
}
template <typename T>
__global__ void __maxnreg__(80) ln_bwd_row_split_addg_v2(const LnBwdArgs a) {
    ln_bwd_row_split_body<T, 2, true>(a);
}

// Stage 1 for any N and alignment: two passes over each row; the partials accumulate in the
// CTA's own workspace rows (each element owned by one thread).
template <typename T, bool VEC, bool ADDG>
__global__ void __launch_bounds__(1024) ln_bwd_stream(const LnBwdArgs a) {
    pdl_enter();  // the stage-2 reductions may be scheduled from now on
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;
    __shared__ float slots[2][2][32];
    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);
    float *pw = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
    float *pb = a.partial + (static_cast<int64_t>(gridDim.x) + blockIdx.x) * a.N;

    auto load = [&](int64_t base, int c, float (&xf)[W], float (&df)[W], float (&wf)[W]) {
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
    };
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * static_cast<int64_t>(a.N);
        const float mu = __ldg(a.mean + row);
        const float rs = __ldg(a.rstd + row);
        float sg = 0.f, sgx = 0.f;
        for (int c = tid; c < nchunk; c += nthr) {
            float xf[W], df[W], wf[W];
            load(base, c, xf, df, wf);
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const float g = df[k] * wf[k];
                sg += g;
                sgx = fmaf(g, (xf[k] - mu) * rs, sgx);
            }
        }
        const float2 t = cta_sum2(sg, sgx, slots[parity]);
        parity ^= 1;
        const float mg = t.x * inv_n, mgx = t.y * inv_n;
        const bool first = (row == blockIdx.x);
        for (int c = tid; c < nchunk; c += nthr) {
            float xf[W], df[W], wf[W], o[W];
            load(base, c, xf, df, wf);
            float gf[W];
            if constexpr (ADDG) {
                if constexpr (VEC) {
                    E::unpack(ld_stream(static_cast<const uint4 *>(a.d_ro) + base / W + c), gf);
                } else {
                    gf[0] = E::load1(a.d_ro, base + c);
                }
            }
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const float xh = (xf[k] - mu) * rs;
                o[k] = rs * (df[k] * wf[k] - mg - xh * mgx);
                if constexpr (ADDG) o[k] += gf[k];
                const int64_t j = static_cast<int64_t>(c) * V + k;
                pw[j] = first ? df[k] * xh : fmaf(df[k], xh, pw[j]);
                pb[j] = first ? df[k] : pb[j] + df[k];
            }
            if constexpr (VEC) {
                st_stream(static_cast<uint4 *>(a.dx) + base / W + c, E::pack(o));
            } else {
                E::store1(a.dx, base + c, o[0]);
            }
        }
    }
}

// ------------------------------------------------------------------------------ dispatch
template <typename T, bool FUSED>
const void *ln_fwd_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_fwd_row_cta<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&ln_fwd_row_cta<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&ln_fwd_row_cta<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&ln_fwd_row_cta<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_WARP:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_fwd_row_warp<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&ln_fwd_row_warp<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&ln_fwd_row_warp<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&ln_fwd_row_warp<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&ln_fwd_stream<T, true, FUSED>)
                         : reinterpret_cast<const void *>(&ln_fwd_stream<T, false, FUSED>);
        default: return nullptr;
    }
}

template <typename T, bool ADDG>
const void *ln_bwd_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_WARP:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_bwd_row_warp<T, 1, ADDG>);
                case 2: return reinterpret_cast<const void *>(&ln_bwd_row_warp<T, 2, ADDG>);
                case 4: return reinterpret_cast<const void *>(&ln_bwd_row_warp<T, 4, ADDG>);
                case 8: return reinterpret_cast<const void *>(&ln_bwd_row_warp<T, 8, ADDG>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_bwd_row_cta<T, 1, ADDG>);
                case 2: return reinterpret_cast<const void *>(&ln_bwd_row_cta<T, 2, ADDG>);
                case 4: return reinterpret_cast<const void *>(&ln_bwd_row_cta<T, 4, ADDG>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_CLUSTER:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_bwd_row_split<T, 1, ADDG>);
                case 2: return ADDG ? reinterpret_cast<const void *>(&ln_bwd_row_split_addg_v2<T>)
                                    : reinterpret_cast<const void *>(&ln_bwd_row_split<T, 2, ADDG>);
                case 4: return reinterpret_cast<const void *>(&ln_bwd_row_split<T, 4, ADDG>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_TMA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&ln_bwd_row_tma<T, 1, ADDG>);
                case 2: return reinterpret_cast<const void *>(&ln_bwd_row_tma<T, 2, ADDG>);
                case 4: return reinterpret_cast<const void *>(&ln_bwd_row_tma<T, 4, ADDG>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&ln_bwd_stream<T, true, ADDG>)
                         : reinterpret_cast<const void *>(&ln_bwd_stream<T, false, ADDG>);
        default: return nullptr;
    }
}

template <typename T>
cudaError_t launch_ln_fwd(const LnFwdArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = a.res ? ln_fwd_kernel_ptr<T, true>(l) : ln_fwd_kernel_ptr<T, false>(l);
    if (!k) return cudaErrorInvalidConfiguration;
    LnFwdArgs args = a;
    void *params[] = {&args};
    return enqueue(k, l, 0, l.variant == RRN_VARIANT_ROW_CTA || l.variant == RRN_VARIANT_ROW_WARP, params, stream);
}

// Stage 1, then stage 2 twice (dw from the first workspace half, db from the second).
template <typename T>
cudaError_t launch_ln_bwd(const LnBwdArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = a.d_ro ? ln_bwd_kernel_ptr<T, true>(l) : ln_bwd_kernel_ptr<T, false>(l);
    if (!k) return cudaErrorInvalidConfiguration;
    if (l.smem > 0) {
        cudaError_t e = allow_dynamic_smem(k, l.smem);
        if (e != cudaSuccess) return e;
    }
    LnBwdArgs args = a;
    args.stages = l.stages;
    void *params[] = {&args};
    cudaError_t e = enqueue(k, l, l.cluster, false, params, stream);
    if (e != cudaSuccess) return e;
    // dw and db together, from the rows stage 1 wrote: one per CTA, or one per cluster
    const int rows = l.cluster ? l.ctas / l.cluster : l.ctas;
    return launch_dw_reduce(a.partial, a.dw, a.db, rows, a.N, stream);
}

template <typename T>
int occupancy_ln_t(bool bwd, bool flag, const Launch &l) {
    const void *k = bwd ? (flag ? ln_bwd_kernel_ptr<T, true>(l) : ln_bwd_kernel_ptr<T, false>(l))
                        : (flag ? ln_fwd_kernel_ptr<T, true>(l) : ln_fwd_kernel_ptr<T, false>(l));
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
