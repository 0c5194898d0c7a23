// RMSNorm (fused with the residual add when a residual is given) feeding an FP8 E4M3 output with
// one fp32 scale per row - the norm fused with the neighbouring quantisation a following FP8
// GEMM needs (the kind of cross-op fusion a persistent megakernel performs: Machete, "Core
// Ideas"). Per row, in fp32:
//   r = x (+ residual);  rstd = rsqrt(sum(r^2) / N + eps);  y = r * rstd * w
//   amax = max |y|;  scale = amax / 448;  q = e4m3_satfinite_rn(y * (448 / amax))
// (q = 0 and scale = 0 for a row whose y is all zero). residual_out = RN(r) as in the plain op.
// The codes come from CUDA's paired fp32 -> e4m3 conversion with saturation to the finite range.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace rrn {

// rstd from the CTA-wide sum of squares, with the rare rescaled path (see rstd_rescaled).
template <typename Each>
__device__ __forceinline__ float rms_rstd(Each each, float ss, float n_f, float eps,
                                          float (&slots)[2][32], int &parity) {
    if (!needs_rescale(ss)) return rstd_plain(ss, n_f, eps);
    float am = 0.f;
    each([&](float v) { am = fmaxf(am, fabsf(v)); });
    am = cta_max(am, slots[parity]);
    parity ^= 1;
    const int e = rescale_exponent(am);
    float s2 = 0.f;
    each([&](float v) {
        const float t = ldexpf(v, -e);
        s2 = fmaf(t, t, s2);
    });
    s2 = cta_sum(s2, slots[parity]);
    parity ^= 1;
    return rstd_rescaled(s2, n_f, eps, e);
}

// rms_rstd over one warp (a row per warp): the warp-wide sum of squares, shuffles only.
template <typename Each>
__device__ __forceinline__ float rms_rstd_warp(Each each, float ss, float n_f, float eps) {
    if (!needs_rescale(ss)) return rstd_plain(ss, n_f, eps);
    float am = 0.f;
    each([&](float v) { am = fmaxf(am, fabsf(v)); });
    const int e = rescale_exponent(warp_max(am));
    float s2 = 0.f;
    each([&](float v) {
        const float t = ldexpf(v, -e);
        s2 = fmaf(t, t, s2);
    });
    return rstd_rescaled(warp_sum(s2), n_f, eps, e);
}

__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Sum of one float and maximum of another over the CTA, with one barrier (fixed order).
__device__ __forceinline__ float2 cta_sum_max(float s, float m, float (*slots)[32]) {
    s = warp_sum(s);
    m = warp_max(m);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        slots[0][warp] = s;
        slots[1][warp] = m;
    }
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float2 t = make_float2(0.f, 0.f);
    for (int i = 0; i < nwarps; ++i) {
        t.x += slots[0][i];
        t.y = fmaxf(t.y, slots[1][i]);
    }
    return t;
}

// The V codes of one vector, q = e4m3(r * rstd * w * inv), written as one 8- or 4-byte store.
template <int V>
__device__ __forceinline__ void store_codes(uint8_t *dst, const float (&f)[V], const float (&wf)[V],
                                            float rs, float inv) {
    uint16_t h[V / 2];
#pragma unroll
    for (int k = 0; k < V / 2; ++k)
        h[k] = e4m3x2(f[2 * k] * rs * wf[2 * k] * inv, f[2 * k + 1] * rs * wf[2 * k + 1] * inv);
    if constexpr (V == 8) {
        *reinterpret_cast<uint2 *>(dst) =
            make_uint2(h[0] | (static_cast<uint32_t>(h[1]) << 16), h[2] | (static_cast<uint32_t>(h[3]) << 16));
    } else {
        *reinterpret_cast<uint32_t *>(dst) = h[0] | (static_cast<uint32_t>(h[1]) << 16);
    }
}

// Row per CTA (rows in registers; w read through L1, prefetched at the start, under the
// forward's register cap). One CTA-wide step per row gives both sum(r^2) and max|r * w|: as
// rstd > 0 multiplies every y, amax = rstd * max|r * w| (within a rounding or two of the amax
// over the fp32 y values, far inside the scale's tolerance; saturation keeps every code finite).
// Only when some |r * w| overflows fp32 does the row take a second step, for the amax of y.
template <typename T, int VPT, bool FUSED>
__global__ void __maxnreg__(fwd_max_regs(VPT)) quant_row_cta(const QuantArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;  // 8 (bf16) or 4 (fp32) codes per vector: 8 or 4 bytes
    __shared__ float slots[2][2][32];
    __shared__ float rescue_slots[2][32];  // the rare rescaled-rstd path's own reductions
    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);
    const uint4 *w4 = static_cast<const uint4 *>(a.w);

#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) prefetch_l1(w4 + c);
    }
    int parity = 0, rescue_parity = 0;
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
        float ss = 0.f, mw = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                E::unpack(ld_keep(w4 + c), wf);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    ss = fmaf(f[k], f[k], ss);
                    mw = fmaxf(mw, fabsf(f[k] * wf[k]));
                }
            }
        }
        const float2 t = cta_sum_max(ss, mw, slots[parity]);
        parity ^= 1;
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
        const float rs = rms_rstd(each, t.x, n_f, a.eps, rescue_slots, rescue_parity);
        float am = rs * t.y;
        if (!isfinite(t.y)) {
            // rare: some |r * w| beyond the fp32 range while y = r * rstd * w is not - the amax
            // over the y values themselves (a uniform decision: t is the same in every thread)
            float m = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = v * nthr + tid;
                if (c < nvec) {
                    float f[V], wf[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
                    E::unpack(ld_keep(w4 + c), wf);
#pragma unroll
                    for (int k = 0; k < V; ++k) m = fmaxf(m, fabsf(f[k] * rs * wf[k]));
                }
            }
            am = cta_max(m, rescue_slots[rescue_parity]);
            rescue_parity ^= 1;
        }
        const float inv = am > 0.f ? 448.f / am : 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                E::unpack(ld_keep(w4 + c), wf);
                store_codes<V>(static_cast<uint8_t *>(a.q) + (base + c) * V, f, wf, rs, inv);
            }
        }
        if (tid == 0) {
            a.scale[row] = am / 448.f;
            if (a.rstd) a.rstd[row] = rs;
        }
    }
}

// Row per warp, for short rows over many rows (as the forward's fwd_row_warp): w in registers
// (loaded once), the row's sum(r^2) and max|r * w| warp-wide (shuffles, no barrier), rows walked
// with a grid-sized stride; otherwise the arithmetic of quant_row_cta.
template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(256) quant_row_warp(const QuantArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    const int nvec = a.N / V;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
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
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                if (FUSED) rv[v] = ld_stream(static_cast<const uint4 *>(a.res) + base + c);
            }
        }
        float ss = 0.f, mw = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                E::unpack(opaque(wv[v]), wf);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    ss = fmaf(f[k], f[k], ss);
                    mw = fmaxf(mw, fabsf(f[k] * wf[k]));
                }
            }
        }
        ss = warp_sum(ss);
        mw = warp_max(mw);
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
        const float rs = rms_rstd_warp(each, ss, n_f, a.eps);
        float am = rs * mw;
        if (!isfinite(mw)) {
            // rare: some |r * w| beyond the fp32 range - the amax over the y values themselves
            float m = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = v * 32 + lane;
                if (c < nvec) {
                    float f[V], wf[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
                    E::unpack(opaque(wv[v]), wf);
#pragma unroll
                    for (int k = 0; k < V; ++k) m = fmaxf(m, fabsf(f[k] * rs * wf[k]));
                }
            }
            am = warp_max(m);
        }
        const float inv = am > 0.f ? 448.f / am : 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                E::unpack(opaque(wv[v]), wf);
                store_codes<V>(static_cast<uint8_t *>(a.q) + (base + c) * V, f, wf, rs, inv);
            }
        }
        if (lane == 0) {
            a.scale[row] = am / 448.f;
            if (a.rstd) a.rstd[row] = rs;
        }
    }
}

// Rows too wide for one CTA's registers, split over the C CTAs of a thread-block cluster as the
// plain forward's fwd_row_cluster splits them: CTA rank q holds the vectors
// [q * chunk, (q + 1) * chunk) of every row its cluster handles, w in registers. Each CTA's
// sum(r^2) and max|r * w| are exchanged through distributed shared memory (ClusterExchange:
// asynchronous remote stores counted on mbarriers, no cluster barrier per row; every CTA combines
// the C pairs in rank order: the same bits everywhere); the rare paths (rescaled rstd, the amax of y itself when some
// |r * w| overflows) exchange one more value each, as the row-per-CTA kernel reduces one more.
template <typename T, int VPT, bool FUSED>
__global__ void __launch_bounds__(fwd_max_threads(VPT)) quant_row_cluster(const QuantArgs a) {
    pdl_enter();
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
    const float n_f = static_cast<float>(a.N);

    uint4 wv[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
    }
    if (tid == 0) xchg.init();
    cluster_sync();  // every CTA of the cluster runs and has its barriers initialised
    int parity = 0;
    // cluster-wide (sum of the first values, max of the second values)
    auto exchange = [&](float s, float m) {
        return xchg(make_float2(s, m), make_float2(0.f, 0.f),
                    [](float2 u, float2 v) { return make_float2(u.x + v.x, fmaxf(u.y, v.y)); },
                    a.faults);
    };

    const int64_t ncl = cluster_nclusters_x();
    for (int64_t row = cluster_id_x(); row < a.M; row += ncl) {
        const int64_t base = row * nvec;
        {
            // ask L2 for this CTA's slices of the cluster's next row now, so that its loads find
            // them there (16384 x 16384 bf16 with a residual: 334 -> 288 us; the same in the plain
            // forward's cluster kernel measured slower, 321 -> 334 us)
            const int64_t nxt = row + ncl;
            if (tid == 0 && c1 > c0 && nxt < a.M) {
                const int64_t nb = nxt * nvec + c0;
                const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
                prefetch_l2_bulk(static_cast<const uint4 *>(a.x) + nb, bytes);
                if (FUSED) prefetch_l2_bulk(static_cast<const uint4 *>(a.res) + nb, bytes);
            }
        }
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                xv[v] = ld_stream(static_cast<const uint4 *>(a.x) + base + c);
                if (FUSED) rv[v] = ld_stream(static_cast<const uint4 *>(a.res) + base + c);
            }
        }
        float ss = 0.f, mw = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                if (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base + c, E::pack(f));
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    ss = fmaf(f[k], f[k], ss);
                    mw = fmaxf(mw, fabsf(f[k] * wf[k]));
                }
            }
        }
        float2 t = cta_sum_max(ss, mw, slots[parity]);
        parity ^= 1;
        t = exchange(t.x, t.y);
        float rs;
        if (!needs_rescale(t.x)) {
            rs = rstd_plain(t.x, n_f, a.eps);
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
            am = cta_max(am, slots[parity][0]);
            parity ^= 1;
            const int e = rescale_exponent(exchange(0.f, am).y);
            float s2 = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (c0 + v * nthr + tid < c1) {
                    float f[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const float u = ldexpf(f[k], -e);
                        s2 = fmaf(u, u, s2);
                    }
                }
            s2 = cta_sum(s2, slots[parity][0]);
            parity ^= 1;
            rs = rstd_rescaled(exchange(s2, 0.f).x, n_f, a.eps, e);
        }
        float am = rs * t.y;
        if (!isfinite(t.y)) {  // rare: some |r * w| beyond fp32 while y is not (see quant_row_cta)
            float m = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v)
                if (c0 + v * nthr + tid < c1) {
                    float f[V], wf[V];
                    r_of<T, FUSED>(xv[v], rv[v], f);
                    E::unpack(wv[v], wf);
#pragma unroll
                    for (int k = 0; k < V; ++k) m = fmaxf(m, fabsf(f[k] * rs * wf[k]));
                }
            m = cta_max(m, slots[parity][0]);
            parity ^= 1;
            am = exchange(0.f, m).y;
        }
        const float inv = am > 0.f ? 448.f / am : 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float f[V], wf[V];
                r_of<T, FUSED>(xv[v], rv[v], f);
                E::unpack(wv[v], wf);
                store_codes<V>(static_cast<uint8_t *>(a.q) + (base + c) * V, f, wf, rs, inv);
            }
        }
        if (q == 0 && tid == 0) {
            a.scale[row] = am / 448.f;
            if (a.rstd) a.rstd[row] = rs;
        }
    }
    cluster_sync();  // no CTA exits while a peer may still write into its shared memory
}

// Any N and alignment: passes over global memory (sum of squares with max|r * w|, then the
// codes; the rare paths one more each), the row re-read from L2. VEC: 128-bit vectors (rows
// too wide for the cluster split); otherwise one element at a time (odd widths, unaligned
// buffers).
template <typename T, bool VEC, bool FUSED>
__global__ void __launch_bounds__(1024) quant_stream(const QuantArgs a) {
    pdl_enter();
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;  // values per chunk
    __shared__ float slots[2][2][32];
    __shared__ float rescue_slots[2][32];
    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float n_f = static_cast<float>(a.N);

    auto load_r = [&](int64_t base, int c, float (&f)[W]) {
        if constexpr (VEC) {
            const int64_t vi = base / W + c;
            E::unpack(__ldcg(static_cast<const uint4 *>(a.x) + vi), f);
            if constexpr (FUSED) {
                float b[W];
                E::unpack(__ldcg(static_cast<const uint4 *>(a.res) + vi), b);
#pragma unroll
                for (int k = 0; k < W; ++k) f[k] += b[k];
            }
        } else {
            f[0] = E::load1(a.x, base + c);
            if constexpr (FUSED) f[0] += E::load1(a.res, base + c);
        }
    };
    auto load_w = [&](int c, float (&wf)[W]) {
        if constexpr (VEC) E::unpack(ld_keep(static_cast<const uint4 *>(a.w) + c), wf);
        else wf[0] = E::load1(a.w, c);
    };
    int parity = 0, rescue_parity = 0;
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
        float ss = 0.f, mw = 0.f;
        for (int c = tid; c < nchunk; c += nthr) {
            float f[W], wf[W];
            load_r(base, c, f);
            load_w(c, wf);
#pragma unroll
            for (int k = 0; k < V; ++k) {
                ss = fmaf(f[k], f[k], ss);
                mw = fmaxf(mw, fabsf(f[k] * wf[k]));
            }
        }
        const float2 t = cta_sum_max(ss, mw, slots[parity]);
        parity ^= 1;
        const float rs = rms_rstd(each, t.x, n_f, a.eps, rescue_slots, rescue_parity);
        float am = rs * t.y;
        if (!isfinite(t.y)) {  // rare: as in quant_row_cta
            float m = 0.f;
            for (int c = tid; c < nchunk; c += nthr) {
                float f[W], wf[W];
                load_r(base, c, f);
                load_w(c, wf);
#pragma unroll
                for (int k = 0; k < V; ++k) m = fmaxf(m, fabsf(f[k] * rs * wf[k]));
            }
            am = cta_max(m, rescue_slots[rescue_parity]);
            rescue_parity ^= 1;
        }
        const float inv = am > 0.f ? 448.f / am : 0.f;
        for (int c = tid; c < nchunk; c += nthr) {
            float f[W], wf[W];
            load_r(base, c, f);
            load_w(c, wf);
            if constexpr (VEC) {
                if constexpr (FUSED) st_stream(static_cast<uint4 *>(a.res_out) + base / W + c, E::pack(f));
                store_codes<W>(static_cast<uint8_t *>(a.q) + base + static_cast<int64_t>(c) * W, f, wf, rs, inv);
            } else {
                if constexpr (FUSED) E::store1(a.res_out, base + c, f[0]);
                static_cast<uint8_t *>(a.q)[base + c] =
                    static_cast<uint8_t>(e4m3x2(f[0] * rs * wf[0] * inv, 0.f) & 0xff);
            }
        }
        if (tid == 0) {
            a.scale[row] = am / 448.f;
            if (a.rstd) a.rstd[row] = rs;
        }
    }
}

template <typename T, bool FUSED>
const void *quant_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&quant_row_cta<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&quant_row_cta<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&quant_row_cta<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&quant_row_cta<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_CLUSTER:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&quant_row_cluster<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&quant_row_cluster<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&quant_row_cluster<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&quant_row_cluster<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_WARP:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&quant_row_warp<T, 1, FUSED>);
                case 2: return reinterpret_cast<const void *>(&quant_row_warp<T, 2, FUSED>);
                case 4: return reinterpret_cast<const void *>(&quant_row_warp<T, 4, FUSED>);
                case 8: return reinterpret_cast<const void *>(&quant_row_warp<T, 8, FUSED>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&quant_stream<T, true, FUSED>)
                         : reinterpret_cast<const void *>(&quant_stream<T, false, FUSED>);
        default: return nullptr;
    }
}

template <typename T>
cudaError_t launch_quant(const QuantArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = a.res ? quant_kernel_ptr<T, true>(l) : quant_kernel_ptr<T, false>(l);
    if (!k) return cudaErrorInvalidConfiguration;
    QuantArgs args = a;
    void *params[] = {&args};
    return enqueue(k, l, l.variant == RRN_VARIANT_ROW_CLUSTER ? l.cluster : 0,
                   l.variant == RRN_VARIANT_ROW_CTA || l.variant == RRN_VARIANT_ROW_WARP, params, stream);
}

template <typename T>
int occupancy_quant_t(bool fused, const Launch &l) {
    const void *k = fused ? quant_kernel_ptr<T, true>(l) : quant_kernel_ptr<T, false>(l);
    if (!k) return 0;
    if (l.cluster > 0) return max_active_clusters(k, l);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, l.threads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace rrn
