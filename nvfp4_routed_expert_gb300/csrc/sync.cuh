// mbarrier, bulk-copy (TMA, non-tensor) and grid-barrier helpers for sm_103a.
//
// Every wait here is bounded: a wait that runs out returns false and the
// caller records kDevErrTimeout in the layer's status word, drains the copies
// it still has in flight (again with a bound) and returns.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace moe {

constexpr uint32_t kMbarSpinLimit = 1u << 22;     // polls of one mbarrier phase
constexpr uint32_t kBarrierSpinLimit = 1u << 21;  // polls of one grid barrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and add `bytes` to the phase's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout.
static __device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kMbarSpinLimit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i > 1024) __nanosleep(32);
    }
    return false;
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Ask the memory system to bring `bytes` (multiple of 16, 16-byte aligned)
// into L2 without waiting.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Order earlier generic-proxy accesses of shared memory before later
// async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier for a co-resident (cooperatively launched) grid.  The
// counter only grows: barrier number n (0, 1, ...) of a launch waits for
// (n + 1) * gridDim.x arrivals, so it needs no reset inside the launch (the
// host zeroes it before each launch).  Returns false, uniformly for the whole
// CTA, if the wait runs out or another CTA has flagged an error.
__device__ __forceinline__ bool grid_barrier(uint32_t* counter, uint32_t n, uint32_t* err,
                                             uint32_t* s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t target = (n + 1) * gridDim.x;
        // the release orders every write this CTA made before the __syncthreads
        red_release_gpu_add(counter, 1u);
        uint32_t ok = 1;
        for (uint32_t i = 0; ld_relaxed_gpu(counter) < target; ++i) {
            if (i >= kBarrierSpinLimit) {
                atomicOr(err, kDevErrTimeout);
                ok = 0;
                break;
            }
            if ((i & 63u) == 63u && ld_relaxed_gpu(err) != 0) {
                ok = 0;
                break;
            }
            if (i > 4096) __nanosleep(64);
        }
        // acquire: the other CTAs' writes before their arrival are visible from here on
        __threadfence();
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

}  // namespace moe
