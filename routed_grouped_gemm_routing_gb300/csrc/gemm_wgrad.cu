// Instantiations of the weight-gradient GEMMs (SM-pair kernels with the
// gathered operand resident in shared memory): DW1 and DW2.
#include "wgrad_pair.cuh"

namespace moe {

// m.b = dh (box 64 x 64), m.c0 = dW1 [E][H][2I] (box 64 x 32)
int launch_gemm_dw1(const GemmArgs& a, const GemmMaps& m, int, cudaStream_t st) {
    return launch_wgrad_pair<DW1>(a, m.b, m.c0, st);
}

// m.a = aw (box 64 x 64), m.c0 = dW2 [E][I][H] (box 64 x 32)
int launch_gemm_dw2(const GemmArgs& a, const GemmMaps& m, int, cudaStream_t st) {
    return launch_wgrad_pair<DW2>(a, m.a, m.c0, st);
}

// FP32 main-gradient accumulation: m.c0 = main_grad_W1 f32 [E][H][2I] or
// main_grad_W2 f32 [E][I][H] (box 32 x 32), added to by TMA reduce-add
int launch_gemm_dw1_mg(const GemmArgs& a, const GemmMaps& m, int, cudaStream_t st) {
    return launch_wgrad_pair<DW1, true>(a, m.b, m.c0, st);
}
int launch_gemm_dw2_mg(const GemmArgs& a, const GemmMaps& m, int, cudaStream_t st) {
    return launch_wgrad_pair<DW2, true>(a, m.a, m.c0, st);
}

}  // namespace moe
