// Inline-PTX wrappers for the Blackwell asynchronous copy engine (bulk copies completing on a
// shared-memory mbarrier) and bounded mbarrier waits.  Every wait has a time limit read from
// %globaltimer; a wait that runs out reports failure instead of spinning forever.
#pragma once

#include <stdint.h>

#include "../../include/gbfft.h"
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
enum : int { KERR_WAIT_TIMEOUT = 1, KERR_STAGE_ALIGN = 2, KERR_BOUNDS = 3 };
// The status an exec call's error word maps to (a misaligned stage is a CUDA-level failure).
inline int kerr_status(int h) {
    return h == 0                   ? FFT_OK
           : h == KERR_WAIT_TIMEOUT ? FFT_ERR_TIMEOUT
           : h == KERR_BOUNDS       ? FFT_ERR_BOUNDS
                                    : FFT_ERR_CUDA;
}

// ---- checked build ------------------------------------------------------------------------
// Built with -DGBFFT_CHECKED (libgbfft_checked.so), the copy-engine kernels test each run-time
// index of a global access, and each tensor-copy coordinate, against the extent of its buffer or
// tensor before using it.  A failing test records KERR_BOUNDS in *err (the first error kept;
// err may be NULL) and the access is skipped; a skipped load still completes its barrier phase,
// without data, so that no wait runs out.  In the normal build every test compiles away.
#ifdef GBFFT_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

__device__ __forceinline__ bool bounds_fail(int* err) {
    if (err) atomicCAS(err, 0, KERR_BOUNDS);
    return false;
}
// [first, first + count) inside [0, extent)
__device__ __forceinline__ bool check_range(int64_t first, int64_t count, int64_t extent,
                                            int* err) {
    if constexpr (!kChecked) {
        return true;
    } else {
        return (first >= 0 && count >= 0 && first <= extent - count) || bounds_fail(err);
    }
}
// A tensor-copy box of w x h elements of `elem` bytes at (x, y) inside an xext x yext plane,
// with x * elem a multiple of 16 bytes (the copy engine's rule for the innermost coordinate),
// and a third coordinate z in [0, zext).
__device__ __forceinline__ bool check_box(int64_t x, int w, int64_t xext, int64_t y, int h,
                                          int64_t yext, int64_t z, int64_t zext, int elem,
                                          int* err) {
    if constexpr (!kChecked) {
        return true;
    } else {
        return ((x * elem) % 16 == 0 && x >= 0 && x <= xext - w && y >= 0 && y <= yext - h &&
                z >= 0 && z < zext) ||
               bounds_fail(err);
    }
}

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
