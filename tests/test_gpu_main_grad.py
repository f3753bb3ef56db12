"""GPU parity of moe_backward_main_grad (FP32 main-gradient accumulation of
the weight gradients) through the C ABI.

* main_grad_out - main_grad_in against the oracle's dW1 / dW2 with the bar of
  the bf16 weight gradients: the accumulators are not rounded to bf16, but
  their operands dh and aw are bf16 intermediates (stored by the L2 dgrad),
  which moves the largest elements by more than the FP32 form of the bar
  allows (e.g. 0.11 at max|dW1| = 45);
* starting from zero main gradients, the result rounded to bf16 equals
  moe_backward's dW1 / dW2 bit for bit (the same FP32 accumulators);
* a second call adds the same gradient again; an expert with no routed slot
  and T = 0 leave the main gradient untouched; dx and d(topk_weights) equal
  moe_backward's."""
import pytest
import torch

from moe_testlib import GpuRun, compare, f32, oracle_all
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _inputs(shape: LayerShape, seed, empty_expert=None):
    inp = make_layer_inputs(shape, seed=seed, device="cpu")
    if empty_expert is not None:
        idx = inp["topk_idx"]
        idx[idx == empty_expert] = (empty_expert + 1) % shape.E
    return {k: v.cuda() for k, v in inp.items()}


def _main_grad_call(run: GpuRun, inp, mg1, mg2, dx, dw):
    B.moe_backward_main_grad(run.shape, inp["dY"], inp["x"], inp["W1"], inp["W2"], inp["topk_w"], run.route,
                             run.saved, run.bwd, dx, mg1, mg2, dw)


@pytest.mark.parametrize("T,H,I,E,k,seed,empty", [
    (300, 256, 192, 6, 3, 30, None),
    (200, 384, 128, 8, 2, 31, 5),
    (130, 128, 64, 4, 4, 32, None),
])
def test_main_grad_matches_oracle_and_bf16_path(T, H, I, E, k, seed, empty):
    shape = LayerShape("mg", T=T, H=H, I=I, E=E, k=k)
    inp = _inputs(shape, seed, empty)
    run = GpuRun(T, H, I, E, k)
    run.run(inp)  # prologue, forward and the bf16 backward
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(seed)
    mg1_in = (torch.randn(E, H, 2 * I, generator=g) * 0.05).cuda()
    mg2_in = (torch.randn(E, I, H, generator=g) * 0.05).cuda()
    mg1, mg2 = mg1_in.clone(), mg2_in.clone()
    dx = torch.full_like(run.dx, float("nan"))
    dw = torch.full_like(run.dw, float("nan"))
    _main_grad_call(run, inp, mg1, mg2, dx, dw)
    torch.cuda.synchronize()
    assert torch.equal(dx, run.dx) and torch.equal(dw, run.dw)
    ref = oracle_all(inp, E)
    compare("main_grad_W1 delta", f32(mg1 - mg1_in), ref["dW1"])
    compare("main_grad_W2 delta", f32(mg2 - mg2_in), ref["dW2"])
    if empty is not None:
        assert torch.equal(mg1[empty], mg1_in[empty]) and torch.equal(mg2[empty], mg2_in[empty])
    # a second call adds the same gradient once more
    first1, first2 = mg1.clone(), mg2.clone()
    _main_grad_call(run, inp, mg1, mg2, dx, dw)
    torch.cuda.synchronize()
    compare("second delta W1", f32(mg1 - first1), ref["dW1"])
    compare("second delta W2", f32(mg2 - first2), ref["dW2"])
    # from zero: the FP32 accumulators themselves, which round to moe_backward's bf16 dW
    z1 = torch.zeros_like(mg1_in)
    z2 = torch.zeros_like(mg2_in)
    _main_grad_call(run, inp, z1, z2, dx, dw)
    torch.cuda.synchronize()
    assert torch.equal(z1.to(torch.bfloat16), run.dW1)
    assert torch.equal(z2.to(torch.bfloat16), run.dW2)


def test_main_grad_no_tokens_adds_nothing():
    T, H, I, E, k = 0, 128, 64, 4, 2
    run = GpuRun(T, H, I, E, k)
    idx = torch.empty(0, k, dtype=torch.int32, device="cuda")
    B.moe_route_prologue(run.shape, idx, run.route)
    mg1 = torch.randn(E, H, 2 * I, device="cuda")
    mg2 = torch.randn(E, I, H, device="cuda")
    a1, a2 = mg1.clone(), mg2.clone()
    empty_bf = torch.empty(0, H, dtype=torch.bfloat16, device="cuda")
    W1 = torch.randn(E, H, 2 * I, device="cuda").to(torch.bfloat16)
    W2 = torch.randn(E, I, H, device="cuda").to(torch.bfloat16)
    w = torch.empty(0, k, dtype=torch.float32, device="cuda")
    B.moe_backward_main_grad(run.shape, empty_bf, empty_bf, W1, W2, w, run.route, run.saved, run.bwd, empty_bf,
                             mg1, mg2, w)
    torch.cuda.synchronize()
    assert torch.equal(mg1, a1) and torch.equal(mg2, a2)


def test_autograd_wrapper_accumulates_main_grad():
    """moe_layer(..., accumulate_main_grad=True) adds dW to W1.main_grad /
    W2.main_grad (FP32) and leaves W1.grad / W2.grad unset."""
    from routed_grouped_gemm_routing_gb300.layer import moe_layer

    shape = LayerShape("agmg", T=150, H=128, I=128, E=4, k=2)
    inp = _inputs(shape, 33)
    ref = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    ref.run(inp)
    x = inp["x"].clone().requires_grad_(True)
    W1 = inp["W1"].clone().requires_grad_(True)
    W2 = inp["W2"].clone().requires_grad_(True)
    W1.main_grad = torch.zeros(W1.shape, dtype=torch.float32, device="cuda")
    W2.main_grad = torch.zeros(W2.shape, dtype=torch.float32, device="cuda")
    w = inp["topk_w"].clone().requires_grad_(True)
    y = moe_layer(x, W1, W2, inp["topk_idx"], w, accumulate_main_grad=True)
    y.backward(inp["dY"])
    torch.cuda.synchronize()
    assert W1.grad is None and W2.grad is None
    assert torch.equal(x.grad, ref.dx) and torch.equal(w.grad, ref.dw)
    assert torch.equal(W1.main_grad.to(torch.bfloat16), ref.dW1)
    assert torch.equal(W2.main_grad.to(torch.bfloat16), ref.dW2)
