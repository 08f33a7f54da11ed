// Device helpers shared by the kernels: mbarriers, bulk (TMA) copies, bounded
// waits, element conversion and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace pkv {

constexpr int kBlockTokens = 16;          // tokens per cache block the kernels implement
// 2 s: a pipeline wait this long is a fault.  The wait-timeout test builds a
// separate copy of the library with a 1 ms limit (PKV_WAIT_LIMIT_NS).
#ifndef PKV_WAIT_LIMIT_NS
#define PKV_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitLimitNs = PKV_WAIT_LIMIT_NS;

// ---- device error word ------------------------------------------------------
// First fault wins; kernels skip the offending access and carry on, so the
// context stays usable and the host reads the code with pkv_device_error.
__device__ __forceinline__ void flag_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// First key (table index) that a query whose last visible key is `last`
// attends under a sliding window of `window` keys (0: no window): the query
// sees keys max(0, last - window + 1) .. last.
__device__ __forceinline__ int window_first_key(int last, int window) {
    return window > 0 ? max(0, last - window + 1) : 0;
}

// The part of decode split `split` (kSplitTokens keys from split * kSplitTokens)
// that a decode query over `ctx` keys attends under a sliding window: blocks
// [begin, end) of its table, the first attended key `lo` (masked below within
// block lo / kBlockTokens), and how many splits the query's keys span (the
// planner's items start at split lo / kSplitTokens).
struct SplitSpan {
    int begin, end, lo, nsplit;
};
__device__ __forceinline__ SplitSpan split_span(int ctx, int split, int window) {
    constexpr int per = kSplitTokens / kBlockTokens;
    SplitSpan r;
    r.lo = window_first_key(ctx - 1, window);
    r.begin = max(split * per, r.lo / kBlockTokens);
    r.end = min((split + 1) * per, (ctx + kBlockTokens - 1) / kBlockTokens);
    r.nsplit = (ctx - 1) / kSplitTokens - r.lo / kSplitTokens + 1;
    return r;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- shared-memory addresses and mbarriers ----------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive `count` times at once (a barrier that expects several consumers).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, records PKV_DEV_WAIT_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            flag_error(err, PKV_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA, tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completing on `bar` with
// `bytes` of transaction count.  src, dst 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- dynamic work units -------------------------------------------------------
// A CTA's producer warp takes work units from a global ticket and hands them to
// the CTA's consumer warps through a 4-deep queue in shared memory, so CTAs that
// start late (because other kernels held their SM) simply find less work.
struct UnitQueue {
    int32_t unit[4];
    int32_t current;          // unit the consumer warps are on
    int32_t pad;
    uint64_t ready[4];        // producer -> consumers
    uint64_t empty[4];        // consumers -> producer
};

__device__ __forceinline__ void uq_init(UnitQueue* q) {
    for (int i = 0; i < 4; ++i) {
        mbar_init(&q->ready[i], 1);
        mbar_init(&q->empty[i], 1);
    }
}

// Producer warp (all lanes): the unit of step k, or -1 when the ticket is
// exhausted or a wait failed; published to the consumers either way.  The
// ticket for step k + 1 is taken here too and kept in `next` (lane 0), so the
// atomic's latency hides behind the issue of step k's copies.  Start with
// next = uq_first_ticket(...).
__device__ __forceinline__ int uq_first_ticket(int* ticket, int lane) {
    return lane == 0 ? atomicAdd(ticket, 1) : 0;
}
__device__ __forceinline__ int uq_produce(UnitQueue* q, uint32_t k, int& next, int* ticket,
                                          int n_units, int lane, int* err, bool& ok) {
    ok = ok && __all_sync(0xffffffffu, mbar_wait(&q->empty[k & 3], ((k >> 2) & 1) ^ 1, err));
    int u = -1;
    if (lane == 0) {
        if (ok && next < n_units) {
            u = next;
            next = atomicAdd(ticket, 1);
        }
        q->unit[k & 3] = u;
        mbar_arrive(&q->ready[k & 3]);
    }
    return __shfl_sync(0xffffffffu, u, 0);
}

// Consumer warps (all `nthreads` threads, named barrier 1): the unit of step k.
// One thread waits for it and publishes it, so every consumer warp sees the same
// sequence of units (and -1 together).
__device__ __forceinline__ int uq_consume(UnitQueue* q, uint32_t k, int nthreads, int* err,
                                          bool& ok) {
    if (threadIdx.x == 0) {
        int u = -1;
        if (ok && mbar_wait(&q->ready[k & 3], (k >> 2) & 1, err)) u = q->unit[k & 3];
        q->current = u;
        mbar_arrive(&q->empty[k & 3]);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
    const int u = *reinterpret_cast<volatile int32_t*>(&q->current);
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
    if (u < 0) ok = false;
    return u;
}

// ---- programmatic dependent launch ---------------------------------------------
// Let the next kernel in the stream start while this grid still runs.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grids this one depends on have completed (no-op without PDL).
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- L2 residency of split partials -------------------------------------------
// Split partials are written while the whole KV stream passes through L2; stored
// with an evict-last policy they are still there when the merge kernel reads them.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(float2* p, float2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(v.x), "f"(v.y),
                 "l"(pol)
                 : "memory");
}

// ---- element conversion -------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    // load N consecutive values (N = 2 or 4) from shared memory as fp32
    template <int N>
    __device__ __forceinline__ static void load(const float* p, float (&out)[N]) {
        if constexpr (N == 4) {
            float4 v = *reinterpret_cast<const float4*>(p);
            out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
        } else {
            float2 v = *reinterpret_cast<const float2*>(p);
            out[0] = v.x; out[1] = v.y;
        }
    }
    __device__ __forceinline__ static float store_val(float x) { return x; }
};

template <>
struct Elem<__nv_bfloat16> {
    template <int N>
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&out)[N]) {
        // a bf16 is the high half of an fp32: widening is a shift / mask
        if constexpr (N == 4) {
            uint2 v = *reinterpret_cast<const uint2*>(p);
            out[0] = __uint_as_float(v.x << 16);
            out[1] = __uint_as_float(v.x & 0xffff0000u);
            out[2] = __uint_as_float(v.y << 16);
            out[3] = __uint_as_float(v.y & 0xffff0000u);
        } else {
            uint32_t v = *reinterpret_cast<const uint32_t*>(p);
            out[0] = __uint_as_float(v << 16);
            out[1] = __uint_as_float(v & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static __nv_bfloat16 store_val(float x) {
        return __float2bfloat16_rn(x);
    }
};

}  // namespace pkv
