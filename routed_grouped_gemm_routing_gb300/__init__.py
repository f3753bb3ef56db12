"""GB300-native routed MoE expert layer (dispatch, L1 grouped GEMM, SwiGLU,
L2 grouped GEMM, top-k weighted combine; forward and backward) behind a
C-ABI library built from hand-written sm_103a CUDA kernels.

Importing the package does not load the CUDA library; ``binding.lib()`` does,
and fails loudly when it has not been built.
"""
from .workloads import CONFIGS, LayerShape, make_layer_inputs, make_routing  # noqa: F401
