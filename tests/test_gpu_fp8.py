"""GPU parity of the FP8 dispatch path through the C ABI.

* moe_quantize_fp8: E4M3 bytes and UE8M0 scale bytes bit-exact against the
  oracle's per-token quantization (integer output: exact bar);
* moe_forward_fp8: y within the comparison bar of the oracle's forward on the
  dequantized input, and bit for bit equal to moe_forward run on that
  dequantized input in bf16 (the widened shared-memory operand is the same);
* moe_dequantize_fp8 bit-exact against the oracle's dequantization, and the
  FP8 training step (quantize, FP8 forward, dequantize, backward) equal to
  the bf16 layer on the dequantized input."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import GpuRun, compare, f32, oracle_route, check_tables
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, bf16_bits, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _quantize_gpu(shape, x):
    T, H = x.shape
    q = torch.full((T, H), 0xAA, dtype=torch.uint8, device="cuda")
    sf = torch.full((T, H // 32), 0xAA, dtype=torch.uint8, device="cuda")
    B.moe_quantize_fp8(shape, x, q, sf)
    torch.cuda.synchronize()
    return q, sf


def _x_with_ranges(T, H, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g) * torch.logspace(-4, 3, T).unsqueeze(1)
    x[0, :64] = 0.0                    # all-zero groups
    if T > 2:
        x[1, :32] = 448.0              # amax exactly 448
        x[1, 32:64] = -449.0           # just above
        x[2, 5] = 1e-30                # tiny group
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("T,H", [(1, 64), (257, 512), (64, 7168), (1000, 128)])
def test_quantize_bit_exact(T, H):
    shape = B.shape_of(T, H, 64, 4, 2)
    x = _x_with_ranges(T, H, seed=T + H)
    q, sf = _quantize_gpu(shape, x.cuda())
    rq, rsf = oracle.quantize_fp8(bf16_bits(x))
    assert np.array_equal(sf.cpu().numpy(), rsf), "UE8M0 scales differ from the oracle"
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != rq)
    assert bad.size == 0, f"{len(bad)} E4M3 bytes differ, first at {bad[0]}: {qg[tuple(bad[0])]:#x} vs {rq[tuple(bad[0])]:#x}"


def _dequantized_bf16(q, sf):
    deq = oracle.dequantize_fp8(q, sf)
    return torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("T,H,I,E,k,seed", [
    (300, 256, 192, 6, 3, 40),
    (64, 128, 64, 8, 2, 41),
    (513, 512, 256, 16, 4, 42),
])
def test_forward_fp8_parity(T, H, I, E, k, seed):
    shape = LayerShape("fp8", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}
    s = B.shape_of(T, H, I, E, k)
    q, sf = _quantize_gpu(s, inp["x"])
    xd = _dequantized_bf16(q.cpu().numpy(), sf.cpu().numpy()).cuda()
    # the bf16 path on the dequantized input
    ref_run = GpuRun(T, H, I, E, k)
    ref_run.run(dict(inp, x=xd), backward=False)
    # the FP8 path
    run = GpuRun(T, H, I, E, k)
    run.poison()
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, inp["W1"], inp["W2"], inp["topk_w"], run.route, run.saved, run.y)
    torch.cuda.synchronize()
    check_tables(run, oracle_route(inp, E))
    assert torch.equal(run.y, ref_run.y), "FP8 forward differs from the bf16 forward on the dequantized input"
    # against the oracle on the dequantized input
    x_bits = bf16_bits(xd.cpu())
    y_ref = oracle.forward(x_bits, bf16_bits(inp["W1"].cpu()), bf16_bits(inp["W2"].cpu()),
                           inp["topk_idx"].cpu().numpy().astype(np.int32), inp["topk_w"].cpu().numpy())
    compare("y (fp8 dispatch)", f32(run.y), y_ref)
    # the quantization error itself stays within E4M3's half step
    xf = inp["x"].float().cpu().numpy()
    err = np.abs(xd.float().cpu().numpy() - xf)
    assert np.all(err <= np.abs(xf) * 2.0 ** -4 + 1e-30 + np.repeat(
        np.ldexp(1.0, sf.cpu().numpy().astype(np.int64) - 127), 32, axis=1) * 2.0 ** -10)


@pytest.mark.parametrize("T,H", [(257, 512), (64, 7168)])
def test_dequantize_bit_exact(T, H):
    shape = B.shape_of(T, H, 64, 4, 2)
    x = _x_with_ranges(T, H, seed=3 * T + H)
    q, sf = _quantize_gpu(shape, x.cuda())
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.moe_dequantize_fp8(shape, q, sf, out)
    torch.cuda.synchronize()
    ref = _dequantized_bf16(q.cpu().numpy(), sf.cpu().numpy())
    assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))


def test_fp8_training_step_equals_bf16_on_the_dequantized_input():
    """quantize -> forward_fp8 -> dequantize -> backward gives, bit for bit,
    the bf16 layer's forward and backward on the dequantized input."""
    T, H, I, E, k = 300, 256, 192, 6, 3
    shape = LayerShape("fp8train", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=44, device="cpu").items()}
    s = B.shape_of(T, H, I, E, k)
    q, sf = _quantize_gpu(s, inp["x"])
    run = GpuRun(T, H, I, E, k)
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, inp["W1"], inp["W2"], inp["topk_w"], run.route, run.saved, run.y)
    xd = torch.empty_like(inp["x"])
    B.moe_dequantize_fp8(run.shape, q, sf, xd)
    B.moe_backward(run.shape, inp["dY"], xd, inp["W1"], inp["W2"], inp["topk_w"], run.route, run.saved, run.bwd,
                   run.dx, run.dW1, run.dW2, run.dw)
    ref = GpuRun(T, H, I, E, k)
    ref.run(dict(inp, x=xd))
    torch.cuda.synchronize()
    for a, b in ((run.y, ref.y), (run.dx, ref.dx), (run.dW1, ref.dW1), (run.dW2, ref.dW2), (run.dw, ref.dw)):
        assert torch.equal(a, b)
