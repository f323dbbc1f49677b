// common.cuh - sm_103a building blocks shared by the kernels: mbarrier + bulk-copy (1-D TMA)
// staging with bounded waits, programmatic-dependent-launch controls, byte permutes, dp4a, and
// the status helpers. Internal header (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_grouped.h"

namespace moe {

constexpr int kMaxEntriesPerPass = 4;      // a group's entries are applied 4 at a time
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits give up after ~1 s

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------- programmatic dependent launch
// wait: block until the grids this one depends on have completed and their writes are visible
// (a no-op when the launch carries no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// a hint: bring the 128-byte line holding p into L2 (returns nothing, changes no result; L2 stays
// coherent with later writes to the line, so it may precede pdl_wait)
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// let the next grid in the stream start launching (it still waits for this grid's completion
// before its own pdl_wait returns).
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- shared-memory mbarriers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// make the barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps (up to the hint,
// in ns) until the phase completes instead of spinning and taking issue slots from other warps.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Division of the non-negative ring and item indices by a divisor fixed for the launch (a ring
// depth, chunks or row blocks per row or group): one multiply-high by a reciprocal computed once per CTA instead of a
// division sequence per work item. Exact for every q below 2^32 / (d - 1), far beyond the indices
// a call reaches; d = 1 passes q through.
struct SmallDiv {
    uint32_t m;
    int d;
    __device__ __forceinline__ explicit SmallDiv(int dv)
        : m(dv > 1 ? 0xFFFFFFFFu / static_cast<uint32_t>(dv) + 1u : 0u), d(dv) {}
    __device__ __forceinline__ int div(int q) const {
        return d > 1 ? static_cast<int>(__umulhi(static_cast<uint32_t>(q), m)) : q;
    }
    __device__ __forceinline__ int mod(int q) const { return q - div(q) * d; }
};

// The retries of mbar_wait_bounded, out of line: the first try_wait sleeps until the phase
// completes (or its time hint runs out), so the loop is cold code that need not sit in the callers'
// hot loops.
static __device__ __noinline__ bool mbar_wait_retry(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Wait for phase `parity` of `bar` to complete; false if it has not after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_retry(bar, parity);
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// An L2 cache policy for data read once (the weight stream): its lines are the first evicted,
// so streaming gigabytes of weights does not push the kernels' code and the small, reused
// per-call data (ids, activations, group tables, h rows, counters) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// ---------------------------------------------------------------- integer helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// dp4a with a's bytes unsigned (0..255) and b's signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float h2f_bits(uint32_t h16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16 & 0xffffu)));
}

}  // namespace moe
