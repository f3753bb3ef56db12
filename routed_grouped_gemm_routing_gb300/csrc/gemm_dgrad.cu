// Instantiations of the data-gradient grouped GEMMs (SM-pair kernels): L2
// dgrad (+ SwiGLU^T) and L1 dgrad.
#include "grouped_gemm_2sm.cuh"

namespace moe {

int launch_gemm_l2_dgrad(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L2_DGRAD>(a, m, max_units, st);
}

int launch_gemm_l1_dgrad(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L1_DGRAD>(a, m, max_units, st);
}

}  // namespace moe
