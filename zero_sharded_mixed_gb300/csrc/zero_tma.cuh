// Shared-memory staging by the TMA engine's linear mode, for the kernels that
// stage their streams through a ring of mbarrier-completed stages.
//
// mbarrier: initialised with an arrival count; a phase completes when that
// many arrivals and every expected transaction byte have arrived; a waiter
// passes the parity of the phase it waits for.  cp.async.bulk copies bytes
// from global to this CTA's shared memory and completes them as transactions
// on an mbarrier.  Every wait here is bounded: mbar_wait_bounded gives up after
// `limit` SM cycles and returns false, so that a caller can record the failure
// and stop instead of spinning forever.
#pragma once

#include <cstdint>

namespace zgb {

static __device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

static __device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

static __device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

static __device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

static __device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Waits for the barrier's phase with the given parity; false after `limit`
// SM cycles.
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - start > limit) return false;
    return true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes`
// transactions on the barrier.  dst 16-byte aligned, src 16-byte aligned,
// bytes a multiple of 16.
static __device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace zgb
