// Instantiations of the grouped GEMM engine: DW1 and DW2.
#include "grouped_gemm.cuh"

namespace moe {

int launch_gemm_dw1(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<DW1>(a, m, grid, st);
}

int launch_gemm_dw2(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<DW2>(a, m, grid, st);
}

}  // namespace moe
