// Asynchronous-copy and mbarrier helpers (inline PTX, sm_100+) shared by the
// libgnn kernels: shared-memory mbarriers, bulk (TMA) copies global ->
// shared, and bounded waits.
#pragma once

#include <stdint.h>

namespace gnn {

// Upper bound on one mbarrier wait; beyond it a kernel records
// GNN_ERR_TIMEOUT in the device error word and stops.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t su32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async proxy (TMA)
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

// true once the phase of parity `parity` has completed
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_test, but the thread may sleep in the instruction (up to about
// 20 us) until the phase completes instead of returning at once, so a waiting
// warp does not take issue slots from the others.
__device__ __forceinline__ bool mbar_test_sleep(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of b: false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, uint32_t parity) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_test_sleep(b, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory to this CTA's shared memory, completing on mbarrier bar.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(su32(bar))
        : "memory");
}

// order earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA) accesses of the same shared memory
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace gnn
