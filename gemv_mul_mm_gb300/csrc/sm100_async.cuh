// sm100_async.cuh -- inline-PTX wrappers for mbarriers and bulk (TMA) copies,
// with bounded waits: a wait gives up after ~1 s of spinning, latches
// DEV_ERR_TIMEOUT and reports failure so the kernel can unwind instead of
// hanging the GPU.
#pragma once

#include <cstdint>

#include "qmm_internal.cuh"

namespace qmm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async (TMA / tensor core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Non-blocking probe: true if the phase with the given parity has completed.
// Much cheaper than try_wait when the phase is already complete.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint (ns): the thread may sleep up to that
// long inside the instruction, and wakes when the phase completes.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity. `abort` is a
// shared flag any warp may raise; waiting stops when it is set. Returns false
// on timeout or abort (the timeout is latched into *err and raises *abort).
// The abort flag and the clock are checked every 16 tries only.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (clock64() - t0 > (1ll << 31)) {  // ~1 s at 2 GHz
            atomicOr(err, DEV_ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Bounded wait for waits on a pipeline's critical path: polls with the cheap
// test_wait, napping `ns` nanoseconds between probes when ns > 0 (a thread
// suspended in try_wait wakes up late). The abort flag and the clock are
// checked every 16 probes.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* err,
                                               unsigned ns) {
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i) {
            if (mbar_test_wait(bar, parity)) return true;
            if (ns) __nanosleep(ns);
        }
        if (*abort) return false;
        if (clock64() - t0 > (1ll << 31)) {  // ~1 s at 2 GHz
            atomicOr(err, DEV_ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// 1-D bulk copy global -> shared, completing `bytes` on `bar`. dst/src must
// be 16-byte aligned and `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace qmm
