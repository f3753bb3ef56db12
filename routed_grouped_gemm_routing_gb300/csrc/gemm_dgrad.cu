// Instantiations of the grouped GEMM engine: L2_DGRAD and L1_DGRAD.
#include "grouped_gemm.cuh"

namespace moe {

int launch_gemm_l2_dgrad(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L2_DGRAD>(a, m, grid, st);
}

int launch_gemm_l1_dgrad(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L1_DGRAD>(a, m, grid, st);
}

}  // namespace moe
