// Instantiations of the forward grouped GEMMs (SM-pair kernels): L1 and L2.
#include "grouped_gemm_2sm.cuh"

namespace moe {

int launch_gemm_l1_fwd(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L1_FWD>(a, m, max_units, st);
}

int launch_gemm_l2_fwd(const GemmArgs& a, const GemmMaps& m, int max_units, cudaStream_t st) {
    return launch_gemm_pair<L2_FWD>(a, m, max_units, st);
}

}  // namespace moe
