// Instantiations of the grouped GEMM engine: L2_DGRAD and L1_DGRAD.
#include "grouped_gemm.cuh"

namespace moe {

int launch_gemm_l2_dgrad(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L2_DGRAD>(a, mA, mB, grid, st);
}

int launch_gemm_l1_dgrad(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L1_DGRAD>(a, mA, mB, grid, st);
}

}  // namespace moe
