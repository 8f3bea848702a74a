// Device-side helpers shared by the Q2_0 kernels: the per-device error word,
// mbarrier / TMA / bulk-copy wrappers (inline PTX, sm_100+ forms) and bounded
// waits. Every wait gives up after a time limit, records
// Q2_0_DEVERR_TIMEOUT and lets the kernel return instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q2_0.h"

namespace q2 {

// First-error-wins device error word: err[0] = code, err[1] = info. Kernels
// receive its address as a parameter.
__device__ __forceinline__ void record_error(unsigned long long *err, int code, long long info) {
    unsigned long long prev = atomicCAS(&err[0], 0ull, (unsigned long long)code);
    if (prev == 0ull) atomicExch(&err[1], (unsigned long long)info);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// As mbar_try_wait, but a thread whose phase is not complete is suspended in
// hardware until it completes or about suspend_ns pass, instead of returning
// at once: waiting threads do not take issue slots from their neighbours.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity,
                                                      uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up after
// limit_ns (about one second unless a kernel passes a shorter limit): records
// the timeout (tag identifies the wait) and returns false.
// Between checks the thread backs off for a few tens of nanoseconds, so that a
// waiting warp takes few issue slots from the warps that share its SM
// sub-partition while still waking within ~100 cycles; sleep = true suspends
// in hardware instead (up to a few hundred cycles of wake-up), for waits with
// slack such as a producer ahead of a deep ring.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kWaitSuspendNs = 20000;
constexpr uint32_t kWaitBackoffNs = 32;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned long long *err,
                                          int tag, bool sleep = false,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    while (true) {
        if (sleep) {
            if (mbar_try_wait_suspend(bar, parity, kWaitSuspendNs)) return true;
        } else {
            __nanosleep(kWaitBackoffNs);
            if (mbar_try_wait(bar, parity)) return true;
        }
        if (globaltimer_ns() - t0 > limit_ns) {
            record_error(err, Q2_0_DEVERR_TIMEOUT, tag);
            return false;
        }
    }
}

// Two or three waits whose phases are usually complete by the time they are
// checked: the non-blocking tests are all issued before any result is used, so
// their latencies overlap; a phase not yet complete takes the bounded wait. A
// set *abort flag (read alongside; optional) makes them return false at once.
__device__ __forceinline__ bool mbar_wait2(uint64_t *b1, uint32_t p1, int tag1, uint64_t *b2,
                                           uint32_t p2, int tag2, unsigned long long *err,
                                           uint64_t limit_ns, const volatile int *abort = nullptr) {
    const int ab = abort ? *abort : 0;
    const bool r1 = mbar_test_wait(b1, p1);
    const bool r2 = mbar_test_wait(b2, p2);
    if (ab) return false;
    if (r1 && r2) return true;
    return (r1 || mbar_wait(b1, p1, err, tag1, false, limit_ns)) &&
           (r2 || mbar_wait(b2, p2, err, tag2, false, limit_ns));
}
__device__ __forceinline__ bool mbar_wait3(uint64_t *b1, uint32_t p1, int tag1, uint64_t *b2,
                                           uint32_t p2, int tag2, uint64_t *b3, uint32_t p3,
                                           int tag3, unsigned long long *err, uint64_t limit_ns,
                                           const volatile int *abort = nullptr) {
    const int ab = abort ? *abort : 0;
    const bool r1 = mbar_test_wait(b1, p1);
    const bool r2 = mbar_test_wait(b2, p2);
    const bool r3 = mbar_test_wait(b3, p3);
    if (ab) return false;
    if (r1 && r2 && r3) return true;
    return (r1 || mbar_wait(b1, p1, err, tag1, false, limit_ns)) &&
           (r2 || mbar_wait(b2, p2, err, tag2, false, limit_ns)) &&
           (r3 || mbar_wait(b3, p3, err, tag3, false, limit_ns));
}

// ---------------------------------------------------------------------------
// Bulk copies (TMA engine)
// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tiled tensor copy global -> shared; c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// Small shared-memory loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

}  // namespace q2
