"""GPU parity of the SwiGLU activation clamp (shape.activation_clamp > 0:
both SwiGLU inputs clamped to [-c, c], gradients passing inside only)
against the clamped CPU oracle, with the bar of moe_testlib.compare on
y, dx, dW1, dW2 and d(topk_weights).  Also: a clamp above every
pre-activation gives bit-for-bit the unclamped results, and the autograd
wrapper passes the clamp through."""
import numpy as np
import pytest
import torch

from moe_testlib import GpuRun, compare, f32, oracle_all
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.layer import moe_layer
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _inputs(shape, seed):
    return {k_: v.cuda() for k_, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}


def _outputs(run):
    return dict(y=f32(run.y), dx=f32(run.dx), dW1=f32(run.dW1), dW2=f32(run.dW2), dtopk_w=f32(run.dw))


@pytest.mark.parametrize("T,H,I,E,k,c,seed", [(200, 256, 192, 6, 3, 1.0, 31), (130, 128, 128, 4, 2, 0.25, 32)])
def test_clamped_layer_matches_oracle(T, H, I, E, k, c, seed):
    shape = LayerShape("clamp", T=T, H=H, I=I, E=E, k=k)
    inp = _inputs(shape, seed)
    run = GpuRun(T, H, I, E, k, activation_clamp=c)
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    ref = oracle_all(inp, E, clamp=c)
    got = _outputs(run)
    for name in ("y", "dx", "dW1", "dW2", "dtopk_w"):
        compare(name, got[name], ref[name], bf16_output=name != "dtopk_w")
    # the clamp is active: the unclamped oracle is far from these results
    free = oracle_all(inp, E)
    assert np.abs(free["y"] - ref["y"]).max() > 10 * np.abs(got["y"] - ref["y"]).max()


def test_clamp_above_every_value_is_bitwise_no_clamp():
    shape = LayerShape("clamp_off", T=150, H=128, I=64, E=5, k=2)
    inp = _inputs(shape, 33)
    runs = []
    for c in (0.0, 1e6):
        r = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k, activation_clamp=c)
        r.run(inp)
        torch.cuda.synchronize()
        runs.append(r)
    for name in ("y", "dx", "dW1", "dW2"):
        a, b = getattr(runs[0], name), getattr(runs[1], name)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    assert torch.equal(runs[0].dw.view(torch.int32), runs[1].dw.view(torch.int32))


def test_autograd_passes_the_clamp():
    shape = LayerShape("clamp_ag", T=96, H=128, I=64, E=4, k=2)
    inp = _inputs(shape, 34)
    c = 0.5
    ref = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k, activation_clamp=c)
    ref.run(inp)
    x = inp["x"].clone().requires_grad_(True)
    W1 = inp["W1"].clone().requires_grad_(True)
    W2 = inp["W2"].clone().requires_grad_(True)
    w = inp["topk_w"].clone().requires_grad_(True)
    y = moe_layer(x, W1, W2, inp["topk_idx"].to(torch.int64), w, activation_clamp=c)
    y.backward(inp["dY"])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.y.view(torch.int16))
    assert torch.equal(x.grad.view(torch.int16), ref.dx.view(torch.int16))
    assert torch.equal(W1.grad.view(torch.int16), ref.dW1.view(torch.int16))
