"""GPU parity at the full workload sizes (DeepSeek-V2-Lite-, V3-, wide- and
skewed-V3-shaped layers) in the launch configuration the benchmark times.

The oracle cannot cover every output at these sizes, so it checks what it
can compute one by one: y, dx and d(topk_weights) of sampled tokens (from a
sub-problem holding those tokens and their experts) and the full dW1 / dW2
of sampled experts (most and least loaded, one below block M and one empty
when present, two random others); every token of the V2-Lite-shaped layer,
512 sampled tokens of the larger ones, and a skewed routing sharp enough to
leave experts empty.  Properties that hold at any size cover the rest: routing
tables bit-exact over the whole routing, every output finite, the combine
equal to the slot-ordered FP32 sum of the weighted rows for every token, and
zero weight gradients for experts that got no slot.  At the V3 shape the FP8
forward is checked on whole experts against the oracle's FP8 forward, the
FP32 main-gradient backward bit for bit against the bf16 path, and the
layer with an activation clamp against the clamped oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import (GpuRun, check_a8_against_oracle, check_tables, compare, dequantized_w1, dequantized_w2, f32,
                         oracle_all, oracle_experts, oracle_route, oracle_tokens)
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _pick_experts(counts, rng, heaviest=True, n_random=2):
    """Most-loaded (unless heaviest=False), least-loaded non-empty, one below
    block M, one empty (when the routing has them) and n_random random
    non-empty experts (at most 1024 rows each when the most loaded one is
    left out, to bound the oracle's time)."""
    order = np.argsort(counts, kind="stable")
    nonzero = order[counts[order] > 0]
    picks = [int(order[-1])] if heaviest else []
    picks.append(int(nonzero[0]))
    for cand in (np.nonzero((counts > 0) & (counts < 128))[0], np.nonzero(counts == 0)[0]):
        cand = [int(e) for e in cand if int(e) not in picks]
        if cand:
            picks.append(cand[0])
    cap = np.inf if heaviest else 1024
    rest = [int(e) for e in rng.permutation(len(counts)) if int(e) not in picks and 0 < counts[e] <= cap]
    return picks + rest[:n_random]


# (workload, sampled tokens, weight-gradient experts include the most loaded)
CASES = [("v2lite", 4096, True), ("v3", 512, True), ("skew", 512, True), ("wide", 512, True),
         ("skew_c1", 128, False)]


@pytest.mark.parametrize("name,n_tok,heaviest", CASES)
def test_full_size(name, n_tok, heaviest):
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
    del acc, o

    rng = np.random.default_rng(1234)
    toks = np.sort(rng.choice(T, size=min(n_tok, T), replace=False))
    y_ref, dx_ref, dw_ref = oracle_tokens(inp, E, toks)
    tt = torch.as_tensor(toks, device="cuda")
    report = {}
    compare(f"{name} y[{len(toks)} tokens]", f32(run.y[tt]), y_ref, report=report)
    compare(f"{name} dx[{len(toks)} tokens]", f32(run.dx[tt]), dx_ref, report=report)
    compare(f"{name} dtopk_w[{len(toks)} tokens]", f32(run.dw[tt]), dw_ref, bf16_output=False, report=report)

    exps = _pick_experts(counts, rng, heaviest=heaviest)
    print(name, "experts", exps, "counts", [int(counts[e]) for e in exps])
    dW1_ref, dW2_ref = oracle_experts(inp, E, exps)
    for i, e in enumerate(exps):
        compare(f"{name} dW1[{e}] ({int(counts[e])} rows)", f32(run.dW1[e]), dW1_ref[i], report=report)
        compare(f"{name} dW2[{e}] ({int(counts[e])} rows)", f32(run.dW2[e]), dW2_ref[i], report=report)


def test_full_size_tiny_every_output():
    """The tiny layer (T=64, H=128, I=64, E=8, k=2): every output and
    gradient against the oracle over the whole problem."""
    shape = CONFIGS["tiny"]
    inp = {k_: v.cuda() for k_, v in make_layer_inputs(shape, seed=0, device="cpu").items()}
    run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    check_tables(run, oracle_route(inp, shape.E))
    ref = oracle_all(inp, shape.E)
    for n, got in (("y", run.y), ("dx", run.dx), ("dW1", run.dW1), ("dW2", run.dW2)):
        compare(f"tiny {n}", f32(got), ref[n])
    compare("tiny dtopk_w", f32(run.dw), ref["dtopk_w"], bf16_output=False)


def test_full_size_fp8_forward_and_main_grad():
    """The V3-shaped layer through the two variants.  The FP8 forward (E4M3
    input and weights, block-scaled MMA, a quantized between the GEMMs) on
    whole experts (the most and the least loaded, one random): the E4M3
    rows of a against oracle.forward_fp8 on a sub-problem of that expert's
    slots and its dequantized weights, and the weighted L2 rows o within the
    comparison bar of the oracle's slot outputs; y finite.  The FP32
    main-gradient backward from zero main gradients rounds to the bf16
    weight gradients bit for bit."""
    shape = CONFIGS["v3"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    inp = make_layer_inputs(shape, seed=5, device="cuda")
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
    run8 = GpuRun(T, H, I, E, k)
    B.moe_route_prologue(run8.shape, inp["topk_idx"], run8.route)
    B.moe_forward_fp8(run8.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run8.route, run8.saved, run8.y)
    torch.cuda.synchronize()
    assert torch.isfinite(run8.y).all()
    tab = run8.tables()
    counts, offs, perm = tab["counts"], tab["offs"], tab["perm"]
    L = B.moe_workspace_layout(run8.shape)
    sv = run8.saved
    R = L.rows_cap
    a8 = sv[L.a: L.a + R * I].view(R, I)
    asf = sv[L.a + R * I: L.a + R * I + R * (I // 32)].view(R, I // 32)
    o = sv[L.o: L.o + R * H * 2].view(torch.bfloat16).view(R, H)
    xq, xsf = q.cpu().numpy(), sf.cpu().numpy()
    w = inp["topk_w"].cpu().numpy()
    rng = np.random.default_rng(7)
    order = np.argsort(counts, kind="stable")
    picks = [int(order[-1]), int(order[0]), int(rng.integers(E))]
    per1, per2 = 2 * I * H // 32, H * I // 32
    for e in dict.fromkeys(picks):
        c = int(counts[e])
        rows = np.arange(offs[e], offs[e] + c)
        slots = perm[rows]
        toks, js = slots // k, slots % k
        x_sub = oracle.dequantize_fp8(xq[toks], xsf[toks])
        W1_sub = dequantized_w1(w1q[e:e + 1].cpu().numpy(), w1sf[e * per1:(e + 1) * per1].cpu().numpy(), 1, H,
                                I).double().numpy()
        W2_sub = dequantized_w2(w2q[e:e + 1].cpu().numpy(), w2sf[e * per2:(e + 1) * per2].cpu().numpy(), 1, H,
                                I).double().numpy()
        y_sub, aq, asf_ref = oracle.forward_fp8(x_sub, W1_sub, W2_sub, np.zeros((c, 1), np.int32),
                                                w[toks, js].reshape(c, 1))
        trows = torch.from_numpy(rows).cuda()
        sf_bad, frac, _ = check_a8_against_oracle(a8[trows].cpu().numpy(), asf[trows].cpu().numpy(),
                                                  np.arange(c), aq, asf_ref, 1)
        print(f"v3 fp8 expert {e} ({c} rows): scale bytes differing {sf_bad:.1e}, codes differing {frac:.1e}")
        compare(f"v3 fp8 o rows of expert {e} ({c} rows)", f32(o[trows]), y_sub)
    del w1q, w1sf, w2q, w2sf, run8
    # FP32 main gradients from the bf16 forward's saved activations
    run = GpuRun(T, H, I, E, k)
    run.run(inp)
    mg1 = torch.zeros(E, H, 2 * I, dtype=torch.float32, device="cuda")
    mg2 = torch.zeros(E, I, H, dtype=torch.float32, device="cuda")
    dx = torch.empty_like(run.dx)
    dw = torch.empty_like(run.dw)
    B.moe_backward_main_grad(run.shape, inp["dY"], inp["x"], inp["W1"], inp["W2"], inp["topk_w"], run.route,
                             run.saved, run.bwd, dx, mg1, mg2, dw)
    torch.cuda.synchronize()
    assert torch.equal(dx, run.dx) and torch.equal(dw, run.dw)
    assert torch.equal(mg1.to(torch.bfloat16), run.dW1)
    assert torch.equal(mg2.to(torch.bfloat16), run.dW2)


def _near_clamp(inp, rows_of_expert, c, delta):
    """For each expert e -> token rows r, the boolean [len(r), 2I] of
    pre-activations within delta of +-c (FP32 products of the bf16 inputs by
    torch's matmul, TF32 off): there the kernel's FP32 decision and the
    oracle's FP64 one may fall on either side of the bound, and both are
    correct readings of the clamp."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        out = {}
        for e, r in rows_of_expert.items():
            h = inp["x"][torch.as_tensor(r, device="cuda")].float() @ inp["W1"][e].float()
            out[e] = ((h.abs() - c).abs() < delta).cpu().numpy()
        return out
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def test_full_size_activation_clamp():
    """The V3-shaped layer with the SwiGLU inputs clamped to [-1, 1] (about a
    third of the gate and up values clipped, their gradients masked), against
    the clamped oracle on sub-problems: y, dx and d(topk_weights) of 256
    sampled tokens, dW2 of the most loaded, the least loaded and one random
    expert, and those experts' dW1 columns whose pre-activations all keep a
    margin of 3e-5 from the bound.  Within the margin the kernel's FP32 and
    the oracle's FP64 may decide differently (measured: a few elements per
    million, at most 7e-6 from the bound), and both are correct readings; a
    flipped decision moves a whole column of dW1 (a feature's column depends
    on that feature's decisions only) but dx only within its bar, so those
    columns are checked finite only."""
    shape = CONFIGS["v3"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    c, delta = 1.0, 3e-5
    inp = make_layer_inputs(shape, seed=3, device="cuda")
    run = GpuRun(T, H, I, E, k, activation_clamp=c)
    run.run(inp)
    torch.cuda.synchronize()
    for t in (run.y, run.dx, run.dW1, run.dW2, run.dw):
        assert torch.isfinite(t).all()
    route = oracle_route(inp, E)
    counts = route["counts"]
    rng = np.random.default_rng(99)
    toks = np.sort(rng.choice(T, size=256, replace=False))
    y_ref, dx_ref, dw_ref = oracle_tokens(inp, E, toks, clamp=c)
    tt = torch.as_tensor(toks, device="cuda")
    compare("v3 clamp y", f32(run.y[tt]), y_ref)
    compare("v3 clamp dx", f32(run.dx[tt]), dx_ref)
    compare("v3 clamp dtopk_w", f32(run.dw[tt]), dw_ref, bf16_output=False)
    order = np.argsort(counts, kind="stable")
    exps = list(dict.fromkeys([int(order[-1]), int(order[0]), int(rng.integers(E))]))
    dW1_ref, dW2_ref = oracle_experts(inp, E, exps, clamp=c)
    perm, offs = route["perm"], route["offs"]
    near = _near_clamp(inp, {e: perm[offs[e]: offs[e] + counts[e]] // k for e in exps}, c, delta)
    for i, e in enumerate(exps):
        compare(f"v3 clamp dW2[{e}]", f32(run.dW2[e]), dW2_ref[i])
        cols = ~near[e].any(axis=0)
        print(f"v3 clamp: dW1[{e}] ({int(counts[e])} rows): {cols.sum()} of {2 * I} columns compared")
        assert cols.sum() >= 0.9 * 2 * I
        compare(f"v3 clamp dW1[{e}]", f32(run.dW1[e])[:, cols], dW1_ref[i][:, cols])


def test_full_size_fp8_forward_skewed():
    """The FP8 forward under the skewed routing at the V3 shape: the most
    loaded expert (thousands of rows: many 256-row units of one expert in a
    row, each on accumulator 0) and the least loaded one, their E4M3 rows of
    a against oracle.forward_fp8 on sub-problems of their slots and
    dequantized weights, and their weighted L2 rows o within the comparison
    bar; y finite."""
    shape = CONFIGS["skew"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    inp = make_layer_inputs(shape, seed=0, device="cuda")
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
    run8 = GpuRun(T, H, I, E, k)
    B.moe_route_prologue(run8.shape, inp["topk_idx"], run8.route)
    B.moe_forward_fp8(run8.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run8.route, run8.saved, run8.y)
    torch.cuda.synchronize()
    assert torch.isfinite(run8.y).all()
    tab = run8.tables()
    counts, offs, perm = tab["counts"], tab["offs"], tab["perm"]
    L = B.moe_workspace_layout(run8.shape)
    sv = run8.saved
    R = L.rows_cap
    a8 = sv[L.a: L.a + R * I].view(R, I)
    asf = sv[L.a + R * I: L.a + R * I + R * (I // 32)].view(R, I // 32)
    o = sv[L.o: L.o + R * H * 2].view(torch.bfloat16).view(R, H)
    xq, xsf = q.cpu().numpy(), sf.cpu().numpy()
    w = inp["topk_w"].cpu().numpy()
    order = np.argsort(counts, kind="stable")
    nz = order[counts[order] > 0]
    per1, per2 = 2 * I * H // 32, H * I // 32
    for e in dict.fromkeys([int(order[-1]), int(nz[0])]):
        c = int(counts[e])
        rows = np.arange(offs[e], offs[e] + c)
        slots = perm[rows]
        toks, js = slots // k, slots % k
        x_sub = oracle.dequantize_fp8(xq[toks], xsf[toks])
        W1_sub = dequantized_w1(w1q[e:e + 1].cpu().numpy(), w1sf[e * per1:(e + 1) * per1].cpu().numpy(), 1, H,
                                I).double().numpy()
        W2_sub = dequantized_w2(w2q[e:e + 1].cpu().numpy(), w2sf[e * per2:(e + 1) * per2].cpu().numpy(), 1, H,
                                I).double().numpy()
        y_sub, aq, asf_ref = oracle.forward_fp8(x_sub, W1_sub, W2_sub, np.zeros((c, 1), np.int32),
                                                w[toks, js].reshape(c, 1))
        trows = torch.from_numpy(rows).cuda()
        sf_bad, frac, _ = check_a8_against_oracle(a8[trows].cpu().numpy(), asf[trows].cpu().numpy(),
                                                  np.arange(c), aq, asf_ref, 1)
        print(f"skew fp8 expert {e} ({c} rows): scale bytes differing {sf_bad:.1e}, codes differing {frac:.1e}")
        compare(f"skew fp8 o rows of expert {e} ({c} rows)", f32(o[trows]), y_sub)
