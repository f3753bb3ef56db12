"""GPU parity at the full workload sizes (DeepSeek-V2-Lite-, V3-, wide- and
skewed-V3-shaped layers) in the launch configuration the benchmark times.

The oracle cannot cover every output at these sizes, so it checks what it
can compute one by one: y, dx and d(topk_weights) of sampled tokens (from a
sub-problem holding those tokens and their experts) and the full dW1 / dW2
of sampled experts (most and least loaded, one below block M when present,
random others).  Properties that hold at any size cover the rest: routing
tables bit-exact over the whole routing, every output finite, the combine
equal to the slot-ordered FP32 sum of the weighted rows for every token, and
zero weight gradients for experts that got no slot.  At the V3 shape the FP8
dispatch forward and the FP32 main-gradient backward are also checked bit
for bit against the bf16 path."""
import numpy as np
import pytest
import torch

from moe_testlib import GpuRun, check_tables, compare, f32, oracle_experts, oracle_route, oracle_tokens
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _pick_experts(counts, n, rng):
    order = np.argsort(counts, kind="stable")
    nonzero = order[counts[order] > 0]
    picks = [int(order[-1]), int(nonzero[0])]
    small = np.nonzero((counts > 0) & (counts < 128))[0]
    if len(small):
        picks.append(int(small[0]))
    rest = [e for e in rng.permutation(len(counts)) if e not in picks and counts[e] > 0]
    picks += [int(e) for e in rest[: max(0, n - len(picks))]]
    return picks[:n]


@pytest.mark.parametrize("name,n_tok,n_exp", [("v2lite", 48, 4), ("v3", 6, 3), ("skew", 6, 3), ("wide", 4, 3)])
def test_full_size(name, n_tok, n_exp):
    shape = CONFIGS[name]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    inp = make_layer_inputs(shape, seed=0, device="cuda")
    run = GpuRun(T, H, I, E, k)
    run.dW1.fill_(float("nan"))
    run.dW2.fill_(float("nan"))
    run.run(inp)
    torch.cuda.synchronize()

    # routing tables over the whole routing
    ref_route = oracle_route(inp, E)
    check_tables(run, ref_route)
    counts = ref_route["counts"]

    # every output finite; experts with no slot have zero gradients
    for t in (run.y, run.dx, run.dW1, run.dW2, run.dw):
        assert torch.isfinite(t).all()
    empty = torch.as_tensor(np.nonzero(counts == 0)[0], device="cuda")
    if empty.numel():
        assert torch.all(run.dW1[empty] == 0) and torch.all(run.dW2[empty] == 0)

    # combine: y[t] is the FP32 slot-ordered sum of the token's weighted rows, rounded once
    o = B.saved_tensors(run.shape, run.saved)["o"]
    inv = torch.as_tensor(ref_route["inv"].astype(np.int64), device="cuda").view(T, k)
    acc = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    for j in range(k):
        r = inv[:, j]
        acc += torch.where((r >= 0)[:, None], o[r.clamp(min=0)].float(), torch.zeros((), device="cuda"))
    assert torch.equal(acc.to(torch.bfloat16), run.y)

    rng = np.random.default_rng(1234)
    toks = np.sort(rng.choice(T, size=n_tok, replace=False))
    y_ref, dx_ref, dw_ref = oracle_tokens(inp, E, toks)
    tt = torch.as_tensor(toks, device="cuda")
    report = {}
    compare("y[sampled tokens]", f32(run.y[tt]), y_ref, report=report)
    compare("dx[sampled tokens]", f32(run.dx[tt]), dx_ref, report=report)
    compare("dtopk_w[sampled tokens]", f32(run.dw[tt]), dw_ref, bf16_output=False, report=report)

    exps = _pick_experts(counts, n_exp, rng)
    dW1_ref, dW2_ref = oracle_experts(inp, E, exps)
    et = torch.as_tensor(exps, device="cuda")
    compare("dW1[sampled experts]", f32(run.dW1[et]), dW1_ref, report=report)
    compare("dW2[sampled experts]", f32(run.dW2[et]), dW2_ref, report=report)
    print(name, "experts", exps, "counts", [int(counts[e]) for e in exps])
    for n, r in report.items():
        print(name, n, {q: f"{v:.3e}" for q, v in r.items()})


def test_full_size_fp8_dispatch_and_main_grad():
    """The V3-shaped layer through the two variants, against the bf16 path
    on the same GPU: the FP8-dispatch forward equals the bf16 forward on the
    dequantized input bit for bit, and the FP32 main-gradient backward from
    zero main gradients rounds to the bf16 weight gradients bit for bit."""
    shape = CONFIGS["v3"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    inp = make_layer_inputs(shape, seed=5, device="cuda")
    s = B.shape_of(T, H, I, E, k)
    q = torch.empty(T, H, dtype=torch.uint8, device="cuda")
    sf = torch.empty(T, H // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_fp8(s, inp["x"], q, sf)
    xd = torch.empty_like(inp["x"])
    B.moe_dequantize_fp8(s, q, sf, xd)
    ref = GpuRun(T, H, I, E, k)
    ref.run(dict(inp, x=xd))
    y8 = torch.empty_like(ref.y)
    B.moe_forward_fp8(ref.shape, q, sf, inp["W1"], inp["W2"], inp["topk_w"], ref.route, ref.saved, y8)
    torch.cuda.synchronize()
    assert torch.equal(y8, ref.y)
    # the saved activations are again those of the dequantized input: main-grad backward
    mg1 = torch.zeros(E, H, 2 * I, dtype=torch.float32, device="cuda")
    mg2 = torch.zeros(E, I, H, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(ref.dx)
    dw = torch.empty_like(ref.dw)
    B.moe_backward_main_grad(ref.shape, inp["dY"], xd, inp["W1"], inp["W2"], inp["topk_w"], ref.route, ref.saved,
                             ref.bwd, dx, mg1, mg2, dw)
    torch.cuda.synchronize()
    assert torch.equal(dx, ref.dx) and torch.equal(dw, ref.dw)
    assert torch.equal(mg1.to(torch.bfloat16), ref.dW1)
    assert torch.equal(mg2.to(torch.bfloat16), ref.dW2)
