// Backward kernels of RMSNorm, with a two-stage deterministic dw.
//
// Per row (xhat = x * rstd, g = dy * w, c = sum(g * xhat) / N):
//   dx = rstd * (g - xhat * c)
// and dw = sum over rows of dy * xhat, reduced in two fixed-order stages:
//   stage 1  CTA p owns rows p, p + P, p + 2P, ... (P CTAs; consecutive CTAs work on adjacent
//            rows at any moment, so HBM is read as one stream); each thread keeps the dw partial
//            sums of its own columns in registers across those rows and writes them once to row
//            p of a [P, N] fp32 workspace.
//   stage 2  dw[j] = sum over p of workspace[p, j], in a fixed order (rows p = g, g+G, ...
//            per group g, then the G group sums in order). No atomics anywhere, so dw is
//            bitwise reproducible for a given (M, N, dtype, device).
// The fused op (residual_out = r = x + residual, y = RMSNorm(r) * w) has the same backward with
// the gradient arriving at residual_out added: d_r = dx + d_ro, the gradient with respect to
// both x and residual (template flag ADDG; r is the stored residual_out).
// The pages give the op (Machete "Built-In Areas": RMSNorm and autograd helpers) but no
// backward formula; the one above is the exact derivative of the forward definition.
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tma.cuh"

namespace rrn {

// dx for one row held in registers (x vectors xv, dy vectors dyv; this thread owns vector
// c = v * blockDim.x + threadIdx.x; rs = rstd[row]), and dy * xhat added into this thread's dw
// registers. `after_reduce` runs right after the CTA-wide dot product, when every thread has
// consumed its inputs; when it returns false the row is abandoned.
template <typename T, int VPT, bool ADDG, typename AfterReduce>
__device__ __forceinline__ bool bwd_row_body(const BwdArgs &a, int64_t row, int nvec,
                                             const uint4 (&xv)[VPT], const uint4 (&dyv)[VPT],
                                             const uint4 (&gv)[VPT], const uint4 (&wv)[VPT],
                                             float (&dw)[VPT][Elem<T>::kPerVec],
                                             float (&slots)[2][32], int &parity, float rs,
                                             AfterReduce after_reduce) {
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    float2 dot2 = splat(0.f);  // packed fp32 pairs: half the FMA instructions
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float xf[V], d[V], wf[V];
            E::unpack(xv[v], xf);
            E::unpack(dyv[v], d);
            E::unpack(wv[v], wf);
#pragma unroll
            for (int k = 0; k < V; k += 2) {
                const float2 xh = mul2(pair(xf[k], xf[k + 1]), splat(rs));
                const float2 d2 = pair(d[k], d[k + 1]);
                dot2 = fma2(mul2(d2, pair(wf[k], wf[k + 1])), xh, dot2);
                const float2 w2 = fma2(d2, xh, pair(dw[v][k], dw[v][k + 1]));
                dw[v][k] = w2.x;
                dw[v][k + 1] = w2.y;
            }
        }
    }
    const float dot = cta_sum(dot2.x + dot2.y, slots[parity]);
    parity ^= 1;
    if (!after_reduce()) return false;
    const float cm = dot * (1.f / static_cast<float>(a.N));  // 1 / N is hoisted out of the row loop
    const int64_t base = row * nvec;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * nthr + tid;
        if (c < nvec) {
            float xf[V], d[V], wf[V], o[V];
            E::unpack(xv[v], xf);
            E::unpack(dyv[v], d);
            E::unpack(wv[v], wf);
#pragma unroll
            for (int k = 0; k < V; k += 2) {
                const float2 xh = mul2(pair(xf[k], xf[k + 1]), splat(rs));
                const float2 g = mul2(pair(d[k], d[k + 1]), pair(wf[k], wf[k + 1]));
                const float2 r = mul2(splat(rs), fma2(xh, splat(-cm), g));
                o[k] = r.x;
                o[k + 1] = r.y;
            }
            if constexpr (ADDG) {
                float g[V];
                E::unpack(gv[v], g);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] += g[k];
            }
            st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
        }
    }
    return true;
}

template <typename T, int VPT>
__device__ __forceinline__ void bwd_prologue(const BwdArgs &a, int nvec, uint4 (&wv)[VPT],
                                             float (&dw)[VPT][Elem<T>::kPerVec]) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * blockDim.x + threadIdx.x;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < Elem<T>::kPerVec; ++k) dw[v][k] = 0.f;
    }
}

// This CTA's dw partial sums -> the [P, N] workspace.
// Without a cluster (CLUSTER == false) CTA p writes row p. With one (the kernel launched in
// clusters of C CTAs; `red` is N floats of this CTA's shared memory), the C CTAs of cluster k
// first add their sums through distributed shared memory - CTA q adds column slice q of all C
// CTAs in rank order - and write row k, so stage 2 reads P / C rows.
template <typename T, int VPT, bool CLUSTER>
__device__ __forceinline__ void bwd_store_partial(const BwdArgs &a, int nvec,
                                                  const float (&dw)[VPT][Elem<T>::kPerVec],
                                                  float *red) {
    constexpr int V = Elem<T>::kPerVec;
    if constexpr (!CLUSTER) {
        float *prow = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * blockDim.x + threadIdx.x;
            if (c < nvec) {
                float4 *dst = reinterpret_cast<float4 *>(prow + static_cast<int64_t>(c) * V);
#pragma unroll
                for (int q = 0; q < V / 4; ++q)
                    dst[q] = make_float4(dw[v][4 * q], dw[v][4 * q + 1], dw[v][4 * q + 2], dw[v][4 * q + 3]);
            }
        }
    } else {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * blockDim.x + threadIdx.x;
            if (c < nvec)
#pragma unroll
                for (int k = 0; k < V; ++k) red[c * V + k] = dw[v][k];
        }
        cluster_sync();  // every CTA's sums are in its shared memory
        const int C = static_cast<int>(cluster_nctarank());
        const int q = static_cast<int>(cluster_ctarank());
        const int slice = (a.N + C - 1) / C;
        const int j0 = q * slice;
        const int j1 = min(a.N, j0 + slice);
        float *prow = a.partial + static_cast<int64_t>(cluster_id_x()) * a.N;
        for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
            float t = 0.f;
            for (int r = 0; r < C; ++r) t += ld_cluster_f32(red + j, static_cast<uint32_t>(r));
            prow[j] = t;
        }
        cluster_sync();  // no CTA leaves while a peer still reads its shared memory
    }
}

// Stage 1 for short rows: a row per warp. Warp w of CTA p takes rows p * W + w, then every
// (P * W)-th row after it (W warps a CTA, P CTAs); lane l owns vectors v * 32 + l. The row's dot
// product is warp-wide (shuffles, no barrier per row); each thread adds dy * xhat into its dw
// registers, and at the end the W warps' sums are added in warp order through shared memory
// (N floats of dynamic shared memory) into row p of the workspace, as a row-per-CTA stage 1
// writes it. (Loading the next row before the current row's arithmetic measured slower: its
// registers cost more warps per SM than the overlap gained - 131072 x 512 bf16 82.0 against
// 71.7 us.)
template <typename T, int VPT, bool ADDG>
__global__ void __launch_bounds__(256) bwd_row_warp(const BwdArgs a) {
    pdl_enter();  // stage 2 may be scheduled from now on; it waits for our results
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    extern __shared__ __align__(16) float red[];
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
    float dw[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = v * 32 + lane;
        if (c < nvec) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = 0.f;
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
        const float rs = __ldg(a.rstd + row);
        float2 dot2 = splat(0.f);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float xf[V], d[V], wf[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(opaque(wv[v]), wf);
#pragma unroll
                for (int k = 0; k < V; k += 2) {
                    const float2 xh = mul2(pair(xf[k], xf[k + 1]), splat(rs));
                    const float2 d2 = pair(d[k], d[k + 1]);
                    dot2 = fma2(mul2(d2, pair(wf[k], wf[k + 1])), xh, dot2);
                    const float2 w2 = fma2(d2, xh, pair(dw[v][k], dw[v][k + 1]));
                    dw[v][k] = w2.x;
                    dw[v][k + 1] = w2.y;
                }
            }
        }
        const float cm = warp_sum(dot2.x + dot2.y) * inv_n;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) {
                float xf[V], d[V], wf[V], o[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(opaque(wv[v]), wf);
#pragma unroll
                for (int k = 0; k < V; k += 2) {
                    const float2 xh = mul2(pair(xf[k], xf[k + 1]), splat(rs));
                    const float2 g = mul2(pair(d[k], d[k + 1]), pair(wf[k], wf[k + 1]));
                    const float2 r = mul2(splat(rs), fma2(xh, splat(-cm), g));
                    o[k] = r.x;
                    o[k + 1] = r.y;
                }
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
    // the W warps' sums, added in warp order, then row blockIdx.x of the workspace
    for (int w = 0; w < W; ++w) {
        if (warp == w) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int c = v * 32 + lane;
                if (c < nvec) {
#pragma unroll
                    for (int k = 0; k < V; ++k) red[c * V + k] = w == 0 ? dw[v][k] : red[c * V + k] + dw[v][k];
                }
            }
        }
        __syncthreads();
    }
    float *prow = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;
    for (int j = threadIdx.x; j < a.N; j += blockDim.x) prow[j] = red[j];
}

template <typename T, int VPT, bool ADDG, bool CLUSTER>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) bwd_row_cta(const BwdArgs a) {
    pdl_enter();  // stage 2 may be scheduled from now on; it waits for our results
    constexpr int V = Elem<T>::kPerVec;
    extern __shared__ __align__(16) float red[];  // N floats when CLUSTER
    __shared__ float slots[2][32];
    const int nvec = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const uint4 *dy4 = static_cast<const uint4 *>(a.dy);
    const uint4 *g4 = static_cast<const uint4 *>(a.d_ro);
    const uint4 *x4 = static_cast<const uint4 *>(a.x);

    uint4 wv[VPT];
    float dw[VPT][V];
    bwd_prologue<T, VPT>(a, nvec, wv, dw);

    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const int64_t base = row * nvec;
        uint4 xv[VPT], dyv[VPT], gv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_stream(x4 + base + c);
                dyv[v] = ld_stream(dy4 + base + c);
                if constexpr (ADDG) gv[v] = ld_stream(g4 + base + c);
            }
        }
        // rstd read here, beside the row's loads: prefetching the next row's value costs this
        // kernel registers (and CTAs per SM) that it cannot spare
        bwd_row_body<T, VPT, ADDG>(a, row, nvec, xv, dyv, gv, wv, dw, slots, parity,
                                   __ldg(a.rstd + row), [] { return true; });
    }
    bwd_store_partial<T, VPT, CLUSTER>(a, nvec, dw, red);
}

// Stage 1 fed by the TMA engine: CTA p owns rows p, p + P, ... and keeps a.stages of them (x,
// dy and, fused, d_ro) in flight in a shared-memory ring filled with cp.async.bulk, refilling a
// slot as soon as the CTA-wide dot product of its row is done.
template <typename T, int VPT, bool ADDG, bool CLUSTER>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) bwd_row_tma(const BwdArgs a) {
    pdl_enter();  // stage 2 may be scheduled from now on; it waits for our results
    constexpr int V = Elem<T>::kPerVec;
    constexpr int NT = ADDG ? 3 : 2;  // rows per slot: x, dy (, d_ro)
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

    uint4 wv[VPT];
    float dw[VPT][V];
    bwd_prologue<T, VPT>(a, nvec, wv, dw);

    int parity = 0;
    int64_t k = 0;
    // rstd of the next row is requested one row ahead: the row data already waits in the ring,
    // so a load issued at the top of the row would put one global-memory round trip on every
    // row's critical path
    float rs = ring.nrows > 0 ? __ldg(a.rstd + ring.first) : 0.f;
    for (; k < ring.nrows; ++k) {
        const float rs_next = k + 1 < ring.nrows ? __ldg(a.rstd + ring.first + (k + 1) * ring.stride) : 0.f;
        if (!ring.wait(a.faults)) abort_flag = 1;
        uint4 xv[VPT], dyv[VPT], gv[VPT];
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = v * nthr + tid;
            if (c < nvec) {
                xv[v] = ld_shared_v4(ring.slot(0) + static_cast<size_t>(c) * 16);
                dyv[v] = ld_shared_v4(ring.slot(1) + static_cast<size_t>(c) * 16);
                if constexpr (ADDG) gv[v] = ld_shared_v4(ring.slot(NT - 1) + static_cast<size_t>(c) * 16);
            }
        }
        const bool done = bwd_row_body<T, VPT, ADDG>(a, ring.first + k * ring.stride, nvec, xv, dyv, gv,
                                                     wv, dw, slots, parity, rs, [&] {
            if (abort_flag) return false;
            if (tid == 0 && k + ring.S < ring.nrows) {
                fence_proxy_async();
                ring.issue(k + ring.S, ring.cur);
            }
            return true;
        });
        if (!done) break;
        ring.advance();
        rs = rs_next;
    }
    if (k < ring.nrows) {
        if (tid == 0) ring.drain(k, ring.S);
        if constexpr (!CLUSTER) return;  // the partial row is not written; the fault word tells
        // (in a cluster the peers still wait at the cluster barriers: take part with the sums)
    }
    // Every row is consumed, so the ring (at least N floats: stages x (2 or 3) rows of N
    // elements of >= 2 bytes) is free to hold the cluster reduction's sums.
    __syncthreads();
    bwd_store_partial<T, VPT, CLUSTER>(a, nvec, dw, reinterpret_cast<float *>(ring_buf));
}

// Stage 1 for rows too wide for one CTA's registers, each row split across the C CTAs of a
// thread-block cluster (C = 2..8): CTA rank q owns the vectors [q * chunk, (q + 1) * chunk) of
// every row its cluster handles (chunk = ceil(nvec / C)), holds that slice of x, dy (, d_ro) in
// registers and keeps the dw partial sums of its columns across rows. A row's dot product
// sum(g * xhat) is the sum of the C CTAs' parts, added in rank order after an exchange through
// distributed shared memory (ClusterExchange: asynchronous remote stores counted on mbarriers, no
// cluster barrier in the row loop - a barrier's release would also wait for the previous row's
// dx stores; measured on 8192 x 16384 bf16: 193 -> 175 us, fused 215 -> 177 us). Cluster k owns
// rows k, k + K, ... (K clusters) and writes its dw partial sums - each CTA its column slice - to
// row k of the [K, N] workspace.
template <typename T, int VPT, bool ADDG>
__device__ __forceinline__ void bwd_row_split_body(const BwdArgs &a) {
    pdl_enter();  // stage 2 may be scheduled from now on; it waits for our results
    using E = Elem<T>;
    constexpr int V = E::kPerVec;
    __shared__ float slots[2][32];
    __shared__ float part[2][kMaxCluster];
    __shared__ __align__(8) uint64_t xbar[2];
    ClusterExchange<float, kMaxCluster> exchange(part, xbar);

    const int nvec = a.N / V;
    const int C = static_cast<int>(cluster_nctarank());
    const int q = static_cast<int>(cluster_ctarank());
    const int chunk = (nvec + C - 1) / C;
    const int c0 = q * chunk;
    const int c1 = min(nvec, c0 + chunk);
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);
    const uint4 *x4 = static_cast<const uint4 *>(a.x);
    const uint4 *dy4 = static_cast<const uint4 *>(a.dy);
    const uint4 *g4 = static_cast<const uint4 *>(a.d_ro);
    if (tid == 0) exchange.init();
    cluster_sync();  // every CTA of the cluster runs and has its barriers initialised

    uint4 wv[VPT];
    float dw[VPT][V];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) wv[v] = ld_keep(static_cast<const uint4 *>(a.w) + c);
#pragma unroll
        for (int k = 0; k < V; ++k) dw[v][k] = 0.f;
    }
    int parity = 0;
    const int64_t first = cluster_id_x();
    const int64_t ncl = cluster_nclusters_x();
    float rs_next = first < a.M ? __ldg(a.rstd + first) : 0.f;
    for (int64_t row = first; row < a.M; row += ncl) {
        const float rs = rs_next;  // requested a row ahead
        if (row + ncl < a.M) rs_next = __ldg(a.rstd + row + ncl);
        const int64_t base = row * nvec;
        {
            // ask L2 for this CTA's slices of the cluster's next row now, so that its loads find
            // them there (8192 x 16384 bf16: 174 -> 140 us plain; 4096 x 32768: 185 -> 146 us;
            // two rows ahead measured no better)
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
                xv[v] = ld_stream(x4 + base + c);
                dyv[v] = ld_stream(dy4 + base + c);
                if constexpr (ADDG) gv[v] = ld_stream(g4 + base + c);
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            if (c0 + v * nthr + tid < c1) {
                float xf[V], d[V], wf[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const float xh = xf[k] * rs;
                    dot = fmaf(d[k] * wf[k], xh, dot);
                    dw[v][k] = fmaf(d[k], xh, dw[v][k]);
                }
            }
        }
        dot = cta_sum(dot, slots[parity]);
        parity ^= 1;
        const float cm = exchange(dot, 0.f, [](float u, float v) { return u + v; }, a.faults) * inv_n;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int c = c0 + v * nthr + tid;
            if (c < c1) {
                float xf[V], d[V], wf[V], o[V];
                E::unpack(xv[v], xf);
                E::unpack(dyv[v], d);
                E::unpack(wv[v], wf);
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] = rs * (d[k] * wf[k] - (xf[k] * rs) * cm);
                if constexpr (ADDG) {
                    float g[V];
                    E::unpack(gv[v], g);
#pragma unroll
                    for (int k = 0; k < V; ++k) o[k] += g[k];
                }
                st_stream(static_cast<uint4 *>(a.dx) + base + c, E::pack(o));
            }
        }
    }
    float *prow = a.partial + first * a.N;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int c = c0 + v * nthr + tid;
        if (c < c1) {
            float4 *dst = reinterpret_cast<float4 *>(prow + static_cast<int64_t>(c) * V);
#pragma unroll
            for (int k = 0; k < V / 4; ++k)
                dst[k] = make_float4(dw[v][4 * k], dw[v][4 * k + 1], dw[v][4 * k + 2], dw[v][4 * k + 3]);
        }
    }
    cluster_sync();  // no CTA leaves while a peer's remote stores may still be on their way to it
}

// The split-row kernel without and with the gradient at residual_out. The latter, at 4 vectors
// a thread, is compiled for 2 resident CTAs of 256 threads (at most 128 registers): it then fits
// with no spills, 4 CTAs of 128 threads per SM instead of 3 at 164 registers (8192 x 16384 bf16:
// 172 -> 166 us; 4096 x 32768: 181 -> 168 us). The plain kernel keeps the compiler's allocation
// (128 at 4 vectors; asking for 2 CTAs gave 123 and ran 2 % slower).
template <typename T, int VPT>
__global__ void __launch_bounds__(bwd_max_threads(VPT)) bwd_row_split(const BwdArgs a) {
    bwd_row_split_body<T, VPT, false>(a);
}
template <typename T, int VPT>
__global__ void __launch_bounds__(bwd_max_threads(VPT), VPT == 4 ? 2 : 1) bwd_row_split_addg(const BwdArgs a) {
    bwd_row_split_body<T, VPT, true>(a);
}

// Two passes over each row (any N, any alignment); the dw partials live in the CTA's own
// workspace row instead of registers. Each workspace element is owned by one thread.
template <typename T, bool VEC, bool ADDG>
__global__ void __launch_bounds__(1024) bwd_stream(const BwdArgs a) {
    pdl_enter();  // stage 2 may be scheduled from now on; it waits for our results
    using E = Elem<T>;
    constexpr int W = E::kPerVec;
    constexpr int V = VEC ? W : 1;
    __shared__ float slots[2][32];

    const int nchunk = a.N / V;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const float inv_n = 1.f / static_cast<float>(a.N);
    float *prow = a.partial + static_cast<int64_t>(blockIdx.x) * a.N;

    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
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
        const float cm = dot * inv_n;
        const bool first = (row == blockIdx.x);
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
            if constexpr (ADDG) {
                float gf[W];
                if constexpr (VEC) {
                    E::unpack(ld_stream(static_cast<const uint4 *>(a.d_ro) + base / W + c), gf);
                } else {
                    gf[0] = E::load1(a.d_ro, base + c);
                }
#pragma unroll
                for (int k = 0; k < V; ++k) o[k] += gf[k];
            }
            if constexpr (VEC) {
                st_stream(static_cast<uint4 *>(a.dx) + base / W + c, E::pack(o));
            } else {
                E::store1(a.dx, base + c, o[0]);
            }
        }
    }
}

// Group g's share of stage 2: acc += src[p * N] for p = p0, p0 + G, ... < P, in that order, U
// loads issued before the first addition of each chunk (so a thread waits for memory about once
// per U rows), the last chunk predicated.
template <int U, int G>
__device__ __forceinline__ float dw_column_sum(const float *src, int p0, int P, int N) {
    float acc = 0.f;
    for (; p0 < P; p0 += U * G) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u * G;
            v[u] = p < P ? src[static_cast<int64_t>(p) * N] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (p0 + u * G < P) acc += v[u];
    }
    return acc;
}

// Stage 2: dw[j] = sum_p partial[p, j]. A CTA covers 32 consecutive columns with
// G = THREADS / 32 row groups (one warp each); group g adds rows p = g, g + G, g + 2G, ...
// in that order (chunks of 16 loads when a group has at most 16 rows, else of 48: predicated-off
// loads still take issue slots; 8192 x 16384 bf16, 148 rows of partial sums: 12.0 -> 6.5 us in
// ncu) - then one warp adds the G group sums in group order. The order depends only on (P, N),
// so dw is reproducible.
// blockIdx.y selects one of two [P, N] blocks of partial sums (the second, reduced into out1,
// follows the first), so that LayerNorm's dw and db reductions run in one launch.
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
    bwd_dw_reduce(const float *__restrict__ partial, float *__restrict__ out0,
                  float *__restrict__ out1, int P, int N) {
    pdl_enter();  // stage 1 has finished and its partial sums are visible
    constexpr int G = THREADS / 32;
    __shared__ float sums[G][33];
    const int lane = threadIdx.x & 31;
    const int grp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    float *dw = blockIdx.y ? out1 : out0;
    float acc = 0.f;
    if (col < N) {
        const float *src = partial + static_cast<int64_t>(blockIdx.y) * P * N + col;
        acc = P <= 16 * G ? dw_column_sum<16, G>(src, grp, P, N) : dw_column_sum<48, G>(src, grp, P, N);
    }
    sums[grp][lane] = acc;
    __syncthreads();
    if (grp == 0 && col < N) {
        float t = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) t += sums[g][lane];
        dw[col] = t;
    }
}

template <typename T, bool ADDG>
const void *bwd_kernel_ptr(const Launch &l) {
    switch (l.variant) {
        case RRN_VARIANT_ROW_CTA:
            switch (l.vpt * 2 + (l.cluster ? 1 : 0)) {
                case 2: return reinterpret_cast<const void *>(&bwd_row_cta<T, 1, ADDG, false>);
                case 3: return reinterpret_cast<const void *>(&bwd_row_cta<T, 1, ADDG, true>);
                case 4: return reinterpret_cast<const void *>(&bwd_row_cta<T, 2, ADDG, false>);
                case 5: return reinterpret_cast<const void *>(&bwd_row_cta<T, 2, ADDG, true>);
                case 8: return reinterpret_cast<const void *>(&bwd_row_cta<T, 4, ADDG, false>);
                case 9: return reinterpret_cast<const void *>(&bwd_row_cta<T, 4, ADDG, true>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_WARP:
            switch (l.vpt) {
                case 1: return reinterpret_cast<const void *>(&bwd_row_warp<T, 1, ADDG>);
                case 2: return reinterpret_cast<const void *>(&bwd_row_warp<T, 2, ADDG>);
                case 4: return reinterpret_cast<const void *>(&bwd_row_warp<T, 4, ADDG>);
                case 8: return reinterpret_cast<const void *>(&bwd_row_warp<T, 8, ADDG>);
                default: return nullptr;
            }
        case RRN_VARIANT_STREAM:
            return l.vec ? reinterpret_cast<const void *>(&bwd_stream<T, true, ADDG>)
                         : reinterpret_cast<const void *>(&bwd_stream<T, false, ADDG>);
        case RRN_VARIANT_ROW_CLUSTER:
            switch (l.vpt) {
                case 1: return ADDG ? reinterpret_cast<const void *>(&bwd_row_split_addg<T, 1>)
                                    : reinterpret_cast<const void *>(&bwd_row_split<T, 1>);
                case 2: return ADDG ? reinterpret_cast<const void *>(&bwd_row_split_addg<T, 2>)
                                    : reinterpret_cast<const void *>(&bwd_row_split<T, 2>);
                case 4: return ADDG ? reinterpret_cast<const void *>(&bwd_row_split_addg<T, 4>)
                                    : reinterpret_cast<const void *>(&bwd_row_split<T, 4>);
                default: return nullptr;
            }
        case RRN_VARIANT_ROW_TMA:
            switch (l.vpt * 2 + (l.cluster ? 1 : 0)) {
                case 2: return reinterpret_cast<const void *>(&bwd_row_tma<T, 1, ADDG, false>);
                case 3: return reinterpret_cast<const void *>(&bwd_row_tma<T, 1, ADDG, true>);
                case 4: return reinterpret_cast<const void *>(&bwd_row_tma<T, 2, ADDG, false>);
                case 5: return reinterpret_cast<const void *>(&bwd_row_tma<T, 2, ADDG, true>);
                case 8: return reinterpret_cast<const void *>(&bwd_row_tma<T, 4, ADDG, false>);
                case 9: return reinterpret_cast<const void *>(&bwd_row_tma<T, 4, ADDG, true>);
                default: return nullptr;
            }
        default: return nullptr;
    }
}

template <typename T>
const void *bwd_kernel_ptr_any(bool add_grad, const Launch &l) {
    return add_grad ? bwd_kernel_ptr<T, true>(l) : bwd_kernel_ptr<T, false>(l);
}

// Stage 2 on the stream, launched with programmatic stream serialisation so that it is
// scheduled while stage 1 drains (it waits for stage 1 inside the kernel). out1 non-NULL: a
// second [P, N] block after the first is reduced into it by the same launch.
inline cudaError_t launch_dw_reduce(const float *partial, float *out0, float *out1, int P, int N,
                                    cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + 31) / 32, out1 ? 2 : 1);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bwd_dw_reduce<kReduceThreads>, partial, out0, out1, P, N);
}

// Stage 1 on l.ctas CTAs (in clusters of l.cluster when set), then stage 2 over the workspace
// rows stage 1 wrote (one per CTA, or one per cluster), on one stream.
template <typename T>
cudaError_t launch_bwd(const BwdArgs &a, const Launch &l, cudaStream_t stream) {
    const void *k = bwd_kernel_ptr_any<T>(a.d_ro != nullptr, l);
    if (!k) return cudaErrorInvalidConfiguration;
    if (l.smem > 0) {
        cudaError_t e = allow_dynamic_smem(k, l.smem);
        if (e != cudaSuccess) return e;
    }
    BwdArgs args = a;
    args.stages = l.stages;
    void *params[] = {&args};
    cudaError_t e = enqueue(k, l, l.cluster, false, params, stream);
    if (e != cudaSuccess) return e;
    return launch_dw_reduce(a.partial, a.dw, nullptr, l.cluster ? l.ctas / l.cluster : l.ctas, a.N,
                            stream);
}

template <typename T>
int occupancy_bwd_t(bool add_grad, const Launch &l) {
    const void *k = bwd_kernel_ptr_any<T>(add_grad, l);
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
