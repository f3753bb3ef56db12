"""GPU parity over a seeded sweep of random small layer shapes, each checked
against the oracle over every output: T, H (multiple of 64), I (multiple of
64), E and k drawn at random, so that expert groups, feature tails, chunk
splits (experts of more than 256 rows) and empty experts fall in ways the
hand-picked cases do not.  The FP8 forward gets its own sweep (H and I
multiples of 128) against oracle.forward_fp8 on the dequantized operands."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import (GpuRun, check_a8_against_oracle, check_tables, compare, dequantized_w1, dequantized_w2, f32,
                         oracle_all, oracle_route)
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _shapes(seed, n, mult):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.choice([1, 3, 5, 8, 16, 33]))
        k = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(1, 700))
        H = mult * int(rng.integers(1, 512 // mult + 1))
        I = mult * int(rng.integers(1, 384 // mult + 1))
        out.append((T, H, I, E, k, int(rng.integers(1 << 30))))
    return out


@pytest.mark.parametrize("T,H,I,E,k,seed", _shapes(2026, 8, 64))
def test_random_shape_forward_backward(T, H, I, E, k, seed):
    shape = LayerShape("sweep", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}
    run = GpuRun(T, H, I, E, k)
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    check_tables(run, oracle_route(inp, E))
    ref = oracle_all(inp, E)
    for n, got in (("y", run.y), ("dx", run.dx), ("dW1", run.dW1), ("dW2", run.dW2)):
        compare(f"{(T, H, I, E, k)} {n}", f32(got), ref[n])
    compare(f"{(T, H, I, E, k)} dtopk_w", f32(run.dw), ref["dtopk_w"], bf16_output=False)


@pytest.mark.parametrize("T,H,I,E,k,seed", _shapes(2027, 5, 128))
def test_random_shape_fp8_forward(T, H, I, E, k, seed):
    shape = LayerShape("sweep8", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}
    s = B.shape_of(T, H, I, E, k)
    q = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    sf = torch.empty(T, H // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_fp8(s, inp["x"], q, sf)
    w1q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device="cuda")
    w1sf = torch.empty(E * 2 * I * H // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_weights_fp8(s, inp["W1"], w1q, w1sf)
    w2q = torch.empty(E, H, I, dtype=torch.uint8, device="cuda")
    w2sf = torch.empty(E * H * I // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_w2_fp8(s, inp["W2"], w2q, w2sf)
    run = GpuRun(T, H, I, E, k)
    run.poison()
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run.route, run.saved, run.y)
    torch.cuda.synchronize()
    tables = oracle_route(inp, E)
    check_tables(run, tables)
    xd = oracle.dequantize_fp8(q.cpu().numpy(), sf.cpu().numpy())
    W1d = dequantized_w1(w1q.cpu().numpy(), w1sf.cpu().numpy(), E, H, I).double().numpy()
    W2d = dequantized_w2(w2q.cpu().numpy(), w2sf.cpu().numpy(), E, H, I).double().numpy()
    idx = inp["topk_idx"].cpu().numpy().astype(np.int32)
    y_ref, aq, asf_ref = oracle.forward_fp8(xd, W1d, W2d, idx, inp["topk_w"].cpu().numpy())
    L = B.moe_workspace_layout(run.shape)
    R = L.rows_cap
    sv = run.saved.cpu().numpy()
    a8 = sv[L.a: L.a + R * I].reshape(R, I)
    asf = sv[L.a + R * I: L.a + R * I + R * (I // 32)].reshape(R, I // 32)
    check_a8_against_oracle(a8, asf, tables["perm"], aq, asf_ref, k)
    compare(f"{(T, H, I, E, k)} y (fp8)", f32(run.y), y_ref)
