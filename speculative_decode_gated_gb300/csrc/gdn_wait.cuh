// Shared-memory mbarriers and the bounded wait on them: the one place where a
// kernel of this library waits for something another agent (the TMA engine,
// the tensor cores) completes.  A wait gives up after about two seconds of
// %globaltimer time instead of spinning forever; the caller then reports
// GDN_DEVERR_TIMEOUT and returns, so the CUDA context stays usable.
#pragma once

#include <cstdint>

namespace gdn {

constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with parity `parity` to complete; false after ~2 s.
__device__ __noinline__ inline bool wait_parity(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            const unsigned long long now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitNs) {
                return false;
            }
        }
    }
}

// Waits for the phases of two barriers with the same parity; false after ~2 s.
__device__ __noinline__ inline bool wait_parity2(uint32_t bar0, uint32_t bar1, uint32_t parity) {
    return wait_parity(bar0, parity) && wait_parity(bar1, parity);
}

}  // namespace gdn
