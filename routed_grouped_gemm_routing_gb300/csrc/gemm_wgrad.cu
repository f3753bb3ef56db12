// Instantiations of the grouped GEMM engine: DW1 and DW2.
#include "grouped_gemm.cuh"

namespace moe {

int launch_gemm_dw1(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, int grid, cudaStream_t st) {
    return launch_gemm_flavour<DW1>(a, mA, mB, grid, st);
}

int launch_gemm_dw2(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mB, int grid, cudaStream_t st) {
    return launch_gemm_flavour<DW2>(a, mA, mB, grid, st);
}

}  // namespace moe
