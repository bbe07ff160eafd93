// Inline-PTX helpers shared by the libkvsel kernels that use mbarriers, bulk
// async copies (TMA) and bounded waits on sm_100-family GPUs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvsel_internal.h"

namespace kvsel_ptx {

constexpr uint64_t kWaitNs = 1000000000ull;  // every wait gives up after 1 s
constexpr uint32_t kSuspendNs = 20000;       // try_wait may park a thread this long (woken on completion)

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of parity `parity`.  Returns false if this or
// another role of the CTA gave up; a timeout sets KVSEL_DEV_TIMEOUT.
__device__ __noinline__ bool wait_phase(uint64_t* b, uint32_t parity, volatile int* abort_flag, unsigned* err) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(b, parity)) return true;
        if ((i & 15) == 0) {
            if (*abort_flag) return false;
            if (gtimer() - t0 > kWaitNs) {
                *abort_flag = 1;
                atomicOr(err, (unsigned)KVSEL_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: drains a thread's own copies or
// MMAs before the CTA releases its resources and exits.
__device__ __noinline__ void drain_phase(uint64_t* b, uint32_t parity) {
    const uint64_t t0 = gtimer();
    while (!mbar_test(b, parity) && gtimer() - t0 < kWaitNs) {
    }
}

// Non-tensor bulk copy global -> shared, completing on mbarrier `bar`
// (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier 1 over `n` threads that also ANDs a flag across them.
template <int n>
__device__ __forceinline__ bool bar_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(n)
        : "memory");
    return r != 0;
}
template <int n>
__device__ __forceinline__ void bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(n) : "memory");
}

}  // namespace kvsel_ptx
