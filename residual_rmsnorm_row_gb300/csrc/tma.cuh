// Bulk asynchronous copies (TMA engine, cp.async.bulk) and mbarriers, as inline PTX for sm_103a,
// plus the library's device fault word.
//
// Only the non-tensor, non-multicast form is used: one contiguous global row -> one
// shared-memory buffer, completion counted in bytes on an mbarrier. Every wait is bounded (by
// the global nanosecond timer and by an iteration cap); a wait that runs out sets a bit in the
// fault word and returns false, and the caller winds down without waiting forever.
#pragma once

#include <stdint.h>

namespace rrn {

// Bit set in the library's device fault word (passed to kernels as a pointer) when an mbarrier
// wait runs out; the host reads and clears the word with rrn_device_faults().
constexpr unsigned int kFaultWaitTimeout = 1u;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitIters = 1u << 28;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later async-proxy ones
// (bulk copies into the same buffer).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Make freshly initialised mbarriers visible to the async proxy (complete_tx from copies).
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count the current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; on timeout set the fault bit in
// *faults and return false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *faults,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kWaitLimitIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && global_ns() - t0 > limit_ns) break;
    }
    if (faults) atomicOr(faults, kFaultWaitTimeout);
    return false;
}

// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to shared
// memory; completion is reported to `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

}  // namespace rrn

namespace rrn {

// ---------------------------------------------------------------------------------------
// Thread-block clusters: rank, distributed shared memory stores, and the cluster barrier.
// The cluster barrier is a hardware barrier instruction (no polling loop).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Store one float into the shared memory of CTA `rank` of this cluster, at the address that
// `local` has in this CTA, and count its 4 bytes as a completed transaction on that CTA's
// mbarrier at the address `bar` has in this CTA. The store is asynchronous: the receiver, having
// announced the bytes it expects (mbar_arrive_expect_tx), waits on its own mbarrier. No cluster
// barrier (and no release of this thread's other memory operations) is involved.
__device__ __forceinline__ void st_async_cluster_f32(const float *local, uint32_t rank, float v,
                                                     const uint64_t *bar) {
    uint32_t rd, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rd) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(rd),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}

// The same for a pair of floats (8 bytes; both addresses 8-byte aligned).
__device__ __forceinline__ void st_async_cluster_f32x2(const float2 *local, uint32_t rank, float2 v,
                                                       const uint64_t *bar) {
    uint32_t rd, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rd) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(rd),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(rb)
                 : "memory");
}

// All threads of all CTAs of the cluster: release this CTA's prior memory operations (incl.
// remote shared-memory stores) and acquire everyone else's.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One value per CTA combined across the C CTAs of a thread-block cluster, through distributed
// shared memory and without a cluster barrier (whose release would also wait for this thread's
// earlier global stores). In each exchange every CTA stores its value into slot q (its rank) of
// every CTA's buffer with an asynchronous remote store that completes a transaction on the
// receiving CTA's mbarrier; each CTA waits on its own mbarrier for the C values and combines them
// in rank order, so every CTA gets the same bits. Two buffers alternate: a CTA sends the value of
// exchange e + 2 only after it has received every peer's value of exchange e + 1, which each peer
// sends after it has read its buffer of exchange e, so no value is overwritten before it is read.
// Waits are bounded; once one runs out the fault word is set and later exchanges no longer wait
// (their results are invalid). The kernel initialises the barriers (init, one thread) and then
// synchronises the cluster once before the first exchange, and once more before any CTA exits.
template <typename VAL, int MAXC>  // VAL: float or float2
struct ClusterExchange {
    VAL (*part)[MAXC];  // [2][MAXC] in shared memory
    uint64_t *bar;      // [2] mbarriers in shared memory
    int C, q;
    int buf;
    uint32_t phase;     // bit b: the phase parity bar[b] completes next
    bool ok;

    __device__ __forceinline__ ClusterExchange(VAL (*p)[MAXC], uint64_t *b)
        : part(p), bar(b), C(static_cast<int>(cluster_nctarank())),
          q(static_cast<int>(cluster_ctarank())), buf(0), phase(0), ok(true) {}
    // One thread, before the cluster synchronisation that precedes the first exchange.
    __device__ __forceinline__ void init() const {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbarrier_init();
    }
    // Every thread of the CTA: send `mine`; return op(...op(op(seed, v_0), v_1)..., v_{C-1}),
    // the C values combined in rank order.
    template <typename Op>
    __device__ __forceinline__ VAL operator()(VAL mine, VAL seed, Op op, unsigned int *faults) {
        const int tid = threadIdx.x;
        if (tid == 0) mbar_arrive_expect_tx(&bar[buf], static_cast<uint32_t>(C * sizeof(VAL)));
        if (tid < C) {
            if constexpr (sizeof(VAL) == 8)
                st_async_cluster_f32x2(&part[buf][q], static_cast<uint32_t>(tid), mine, &bar[buf]);
            else
                st_async_cluster_f32(&part[buf][q], static_cast<uint32_t>(tid), mine, &bar[buf]);
        }
        if (ok && !mbar_wait(&bar[buf], (phase >> buf) & 1u, faults)) ok = false;
        phase ^= 1u << buf;
        VAL t = seed;
        for (int i = 0; i < C; ++i) t = op(t, part[buf][i]);
        buf ^= 1;
        return t;
    }
};

// A CTA's ring of S shared-memory slots fed by bulk copies. Slot k % S holds row k of the CTA
// (global row first + k * stride, k < nrows) of NT tensors - src[t] + row * row_bytes - and
// completes on the mbarrier full[k % S]. One thread initialises the barriers and issues the
// copies; every thread waits. A slot may be refilled once every thread is done reading it.
// The row being worked on is followed by a cursor (its slot `cur` and the parity `phase` of
// that slot's fill), advanced once per row, so the hot loop divides nothing by S.
template <int NT>
struct RowRing {
    unsigned char *buf;  // S * NT * row_bytes bytes of dynamic shared memory
    uint64_t *full;      // S mbarriers
    const char *src[NT];
    uint32_t row_bytes;
    int S;
    int64_t first, stride, nrows;
    int cur = 0;
    uint32_t phase = 0;

    __device__ __forceinline__ unsigned char *at(int s, int t) const {
        return buf + static_cast<uint32_t>(s * NT + t) * row_bytes;
    }
    // tensor t of the row under the cursor
    __device__ __forceinline__ unsigned char *slot(int t) const { return at(cur, t); }
    // the slot the cursor held one row earlier
    __device__ __forceinline__ int prev() const { return cur == 0 ? S - 1 : cur - 1; }
    __device__ __forceinline__ void advance() {
        if (++cur == S) {
            cur = 0;
            phase ^= 1u;
        }
    }
    // One thread, before the CTA barrier that precedes any use.
    __device__ __forceinline__ void init() const {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbarrier_init();
        fence_proxy_async();
    }
    // One thread: request row k of every tensor into slot s (= k % S). The caller has ordered
    // its own earlier reads of that slot (fence_proxy_async) when the slot is being refilled.
    __device__ __forceinline__ void issue(int64_t k, int s) const {
        uint64_t *bar = &full[s];
        const int64_t off = (first + k * stride) * static_cast<int64_t>(row_bytes);
        mbar_arrive_expect_tx(bar, NT * row_bytes);
#pragma unroll
        for (int t = 0; t < NT; ++t) bulk_g2s(at(s, t), src[t] + off, row_bytes, bar);
    }
    // One thread: fill the ring with the first rows.
    __device__ __forceinline__ void prime() const {
        for (int s = 0; s < S && s < nrows; ++s) issue(s, s);
    }
    // Every thread: wait (bounded) until the row under the cursor has landed; false after a
    // timeout.
    __device__ __forceinline__ bool wait(unsigned int *faults) const {
        return mbar_wait(&full[cur], phase, faults);
    }
    // One thread, after the CTA gave up at row k: let the copies already issued - rows k to
    // k + ahead - 1 - land before the shared memory is released (each wait bounded again).
    __device__ __forceinline__ void drain(int64_t k, int ahead) const {
        for (int64_t j = k; j < nrows && j < k + ahead; ++j)
            (void)mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1), nullptr, 100000000ull);
    }
};

// Load one float from the shared memory of CTA `rank` of this cluster, at the address `local`
// has in this CTA.
__device__ __forceinline__ float ld_cluster_f32(const float *local, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// A hint to bring [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16): no
// completion to wait for, no effect on any value.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

}  // namespace rrn
