// Helpers shared by the grouped-GEMM kernels of the routed MoE layer (the
// row-grouped SM-pair GEMMs and the weight-gradient SM-pair GEMMs).
#pragma once

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

// Every lane of the warp waits; the warp proceeds only if all lanes saw the
// phase complete, so warp-collective instructions never run diverged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Output tensor maps of an epilogue (TMA stores); unused ones are null.
struct OutMaps {
    const CUtensorMap* c0;
    const CUtensorMap* c1;
};

}  // namespace moe
