// Device helpers shared by the RMSNorm kernels: 128-bit vector types per storage dtype,
// cache-hinted loads and stores, and the fp32 warp / CTA sum reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rrn {

// ----------------------------------------------------------------------------------------
// Element types. A "vector" is 16 bytes: 8 bf16 or 4 fp32 values, moved as one uint4
// (one 128-bit LDG/STG per thread, the access width the CuTe DSL skill page's invariants
// P1-P2 derive from the element width).
// ----------------------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    using Storage = uint16_t;

    // Widening bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
    __device__ __forceinline__ static void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(u[i] << 16);
            f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    }
    // One round-to-nearest-even per value.
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
    }
    __device__ __forceinline__ static float load1(const void *p, int64_t i) {
        const uint16_t b = static_cast<const uint16_t *>(p)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ __forceinline__ static void store1(void *p, int64_t i, float v) {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    }
};

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    using Storage = float;

    __device__ __forceinline__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float load1(const void *p, int64_t i) {
        return static_cast<const float *>(p)[i];
    }
    __device__ __forceinline__ static void store1(void *p, int64_t i, float v) {
        static_cast<float *>(p)[i] = v;
    }
};

// r = x (+ residual) in fp32 for one 128-bit vector of packed inputs. Recomputing it is exact
// and cheap, so the kernels keep the row packed (4 registers per vector and tensor) instead of
// holding an fp32 copy across the reduction.
template <typename T, bool FUSED>
__device__ __forceinline__ void r_of(const uint4 &xv, const uint4 &rv,
                                     float (&f)[Elem<T>::kPerVec]) {
    using E = Elem<T>;
    E::unpack(xv, f);
    if constexpr (FUSED) {
        float b[E::kPerVec];
        E::unpack(rv, b);
#pragma unroll
        for (int k = 0; k < E::kPerVec; ++k) f[k] += b[k];
    }
}

// ----------------------------------------------------------------------------------------
// Memory access. Row data is touched exactly once, so it is loaded and stored with the
// streaming (evict-first) hint; the weight vector is re-read by every row and goes through
// the read-only path so it stays cached. Row loads use the coherent path (not .nc) because an
// output may alias an input buffer.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }
__device__ __forceinline__ uint4 ld_keep(const uint4 *p) { return __ldg(p); }
// The same bits, opaque to the compiler: a loop-invariant packed vector passed through this in
// the loop is unpacked there, rather than once before the loop into twice the registers.
__device__ __forceinline__ uint4 opaque(uint4 v) {
    asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
    return v;
}
// Pull a line into L1 ahead of its use, without holding a register for it.
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// ----------------------------------------------------------------------------------------
// Programmatic dependent launch. A kernel calls pdl_allow_dependents() to let the next kernel
// on the stream - when that one was launched with programmatic stream serialisation - be
// scheduled before this one finishes; the dependent kernel calls pdl_wait() before it reads
// anything the first one writes (it returns once the first grid has completed and its memory
// is visible). Without such a launch both are no-ops.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The first statement of every kernel of the library (each may be launched as a programmatic
// dependent of the kernel before it on the stream): let the next kernel be scheduled once every
// CTA of this one is running, then wait until the previous kernel has completed and its memory
// is visible, before any access to global memory. Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_enter() {
    pdl_allow_dependents();
    pdl_wait();
}

// ----------------------------------------------------------------------------------------
// Reductions: butterfly over the warp with shfl_xor (every lane ends with the total), then
// one shared-memory slot per warp, summed by every thread in warp order. The order is fixed,
// so the result is the same on every run and every thread of the CTA sees the same bits.
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// `slots` holds at least blockDim.x / 32 floats. Callers alternate between two slot arrays
// on successive calls so one __syncthreads per call is enough: a slot array is rewritten only
// after every thread has passed the barrier of the call in between.
__device__ __forceinline__ float cta_sum(float v, float *slots) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) slots[warp] = v;
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float t = 0.f;
    for (int i = 0; i < nwarps; ++i) t += slots[i];
    return t;
}

__device__ __forceinline__ float cta_max(float v, float *slots) {
    v = warp_max(v);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) slots[warp] = v;
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    float t = 0.f;
    for (int i = 0; i < nwarps; ++i) t = fmaxf(t, slots[i]);
    return t;
}

// ----------------------------------------------------------------------------------------
// rstd from an fp32 sum of squares. r^2 overflows fp32 once |r| exceeds about 1.8e19 and
// underflows below about 1e-19; then (and for an all-zero row) the kernels take a rare path:
// they rescale the row by 2^-k, with k chosen so the row's largest magnitude lands in [1, 2),
// sum the squares again, and undo the scaling on rstd. The scaling is exact (a power of two).
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ float rstd_plain(float ss, float n, float eps) {
    return rsqrtf(ss / n + eps);
}

__device__ __forceinline__ bool needs_rescale(float ss) {
    return !(ss >= 0x1p-64f && ss <= 3.40282347e38f);
}

// k such that amax * 2^-k is in [1, 2); 0 for a zero, infinite or NaN amax.
__device__ __forceinline__ int rescale_exponent(float amax) {
    if (!(amax > 0.f) || isinf(amax)) return 0;
    int e = 0;
    (void)frexpf(amax, &e);
    return e - 1;
}

// rstd = 1 / sqrt(mean(r^2) + eps) given ss_scaled = sum((r * 2^-k)^2).
__device__ __forceinline__ float rstd_rescaled(float ss_scaled, float n, float eps, int k) {
    const float e2 = ldexpf(eps, -2 * k);
    if (isinf(e2)) return rsqrtf(eps);  // eps outweighs mean(r^2) by more than 2^128
    return ldexpf(rsqrtf(ss_scaled / n + e2), -k);
}

// ------------------------------------------------------------------ packed fp32 pairs
// The fp32x2 add / mul / fma of sm_100-class GPUs: one instruction for two lanes, each lane
// rounded exactly as the scalar fp32 operation would be. Worth it where a kernel's issue rate,
// not its memory traffic, sets the pace (the LayerNorm backward).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 pair(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 splat(float a) { return make_float2(a, a); }

}  // namespace rrn
