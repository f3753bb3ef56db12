// Instantiations of the grouped GEMM engine: L1_FWD and L2_FWD.
#include "grouped_gemm.cuh"

namespace moe {

int launch_gemm_l1_fwd(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L1_FWD>(a, m, grid, st);
}

int launch_gemm_l2_fwd(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
    return launch_gemm_flavour<L2_FWD>(a, m, grid, st);
}

}  // namespace moe
