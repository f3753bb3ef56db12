// Helpers shared by the grouped-GEMM kernels of the routed MoE layer (the
// row-grouped SM-pair GEMMs and the weight-gradient SM-pair GEMMs).
#pragma once

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

// Every lane of the warp waits; the warp proceeds only if all lanes saw the
// phase complete, so warp-collective instructions never run diverged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
    const bool ok = mbar_wait(bar, parity, abort, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded wait: every lane polls and the loop condition is a
// warp vote, so the warp stays converged.  The MMA-issuing warps wait this
// way: after a wait loop run by one diverged thread, each tcgen05.mma that
// follows costs that thread ~100 cycles (measured on this GPU), more than
// the tensor pipe needs for an N = 128 MMA; after a converged wait, an
// elected lane issues at the pipe's rate.  kCluster: acquire at cluster
// scope (barriers that receive arrivals from the other CTA of the pair).
template <bool kCluster>
__device__ __forceinline__ bool warp_wait_uniform(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    auto poll = [&]() -> bool {
        if constexpr (kCluster) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(bar), "r"(parity)
                : "memory");
            return __all_sync(0xffffffffu, ok != 0);
        } else {
            return __all_sync(0xffffffffu, mbar_try_wait(bar, parity));
        }
    };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (poll()) return true;
        if ((it & 63u) == 0) {
            const bool late = global_timer_ns() - t0 > limit_ns;
            if (__any_sync(0xffffffffu, *abort != 0 || late)) {
                if (late) *abort = 1;
                return false;
            }
        }
    }
}

// One lane of a converged warp (the same lane every time the whole warp
// calls it), for issuing tcgen05.mma and tcgen05.commit: a commit tracks
// only the MMAs issued by its own thread.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Output tensor maps of an epilogue (TMA stores); unused ones are null.
struct OutMaps {
    const CUtensorMap* c0;
    const CUtensorMap* c1;
};

}  // namespace moe
