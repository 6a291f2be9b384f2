// Inline-PTX wrappers for the Blackwell asynchronous copy engine (bulk copies completing on a
// shared-memory mbarrier) and bounded mbarrier waits.  Every wait has a time limit read from
// %globaltimer; a wait that runs out reports failure instead of spinning forever.
#pragma once

#include <stdint.h>

#include "launch_cache.cuh"

namespace gbfft {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy shared-memory accesses (made visible to this thread by a barrier)
// before later asynchronous-proxy writes to the same shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global memory to
// this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_smem_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete, for at most limit_ns nanoseconds.
// limit_ns == 0 gives up without polling (a diagnostic hook to exercise the timeout path).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (limit_ns == 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s for draining copies after a timeout


// Error word values written by kernels (read and cleared by fft_plan_check).
enum : int { KERR_WAIT_TIMEOUT = 1, KERR_STAGE_ALIGN = 2 };

// Self-check run once per CTA before its first asynchronous copy: the shared-memory stage must
// start on a 128-byte boundary (copies need 16).  On failure the CTA records KERR_STAGE_ALIGN
// (err may be NULL) and issues nothing.  tma_stage_aligned is the uniform form (every thread
// evaluates it); stage_misaligned is the single-thread form whose result the kernel publishes
// through shared memory across its prologue barrier.
__device__ __forceinline__ bool tma_stage_aligned(const void* stage, int* err) {
    const bool ok = (smem_addr(stage) & 127u) == 0;
    if (!ok && threadIdx.x == 0 && err) atomicExch(err, KERR_STAGE_ALIGN);
    return ok;
}
__device__ __forceinline__ int stage_misaligned(const void* stage, int* err) {
    const bool bad = (smem_addr(stage) & 127u) != 0;
    if (bad && err) atomicExch(err, KERR_STAGE_ALIGN);
    return bad ? 1 : 0;
}

}  // namespace gbfft
