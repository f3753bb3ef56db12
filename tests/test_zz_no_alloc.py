"""The allocation-free inference forward, moe_forward_noalloc.

It serves callers that cannot allocate device memory when they run the
layer (a plugin inside an inference engine that is given no workspace, a
serving loop that must not call cudaMalloc because it can synchronise the
device): routing tables and intermediates live in a static device array
inside the library.  Checked through the C ABI against the workspace-based
moe_route_prologue + moe_forward, with the same tolerance as every other
parity test, on two calls in a row (the second with other routing and
another shape, so stale scratch contents would show), and its size limit is
checked on the host.  This file is collected last on purpose."""
import pytest
import torch

from moe_testlib import GpuRun, compare, f32
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _forward_both(shape, seed):
    inp = {k: v.cuda() for k, v in make_layer_inputs(shape, seed=seed, device="cpu", with_grad_out=False).items()}
    ref = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    ref.run(inp, backward=False)
    y = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_forward_noalloc(B.shape_of(shape.T, shape.H, shape.I, shape.E, shape.k), inp["x"], inp["W1"], inp["W2"],
                          inp["topk_idx"], inp["topk_w"], y)
    torch.cuda.synchronize()
    return y, ref.y


def test_noalloc_forward_matches_workspace_forward_twice():
    first = LayerShape("noalloc_a", T=64, H=128, I=64, E=8, k=2)
    second = LayerShape("noalloc_b", T=150, H=256, I=192, E=6, k=3)
    for shape, seed in ((first, 0), (second, 1)):
        y, y_ref = _forward_both(shape, seed)
        compare(f"y ({shape.name})", f32(y), f32(y_ref))
        assert torch.equal(y, y_ref)  # same kernels, same order: identical bits


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    s = B.shape_of(4096, 2048, 1408, 64, 6)  # needs ~410 MB of scratch
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    L = B.lib()
    fn = L.moe_forward_noalloc
    fn.argtypes = [B.ctypes.POINTER(B.MoeShape)] + [B.ctypes.c_void_p] * 7
    fn.restype = B.ctypes.c_int
    p = dummy.data_ptr()
    assert fn(B.ctypes.byref(s), p, p, p, p, p, p, None) == B.MOE_EUNSUPPORTED  # rejected before any launch
    assert "static scratch" in B.moe_last_error()
