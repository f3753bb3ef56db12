"""GPU parity of the FP8 path through the C ABI.

* moe_quantize_fp8 and moe_quantize_weights_fp8: E4M3 bytes and UE8M0 scale
  bytes bit-exact against the oracle's quantization (integer output: exact
  bar; the weights' scales read back from the kernel's atom layout);
* moe_quantize_w2_fp8: the same for W2;
* moe_forward_fp8 (block-scaled tensor-core MMA on E4M3 operands in both
  GEMMs, the SwiGLU output quantized between them): its E4M3 activations
  against the oracle's (a few codes one step apart, where the FP32 and the
  float64 a round to different sides of a midpoint), y within the
  comparison bar of the L2 contraction of its own E4M3 activations (exact
  operands) and of oracle.forward_fp8 on the dequantized operands;
* moe_dequantize_fp8 bit-exact against the oracle's dequantization."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import (GpuRun, check_a8_against_oracle, check_tables, compare, dequantized_w1, dequantized_w2,
                         f32, oracle_route, unpack_w1_atoms, unpack_w2_atoms)
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


def _quantize_w1_gpu(shape, W1):
    E, H, I2 = W1.shape
    q = torch.full((E, I2, H), 0xAA, dtype=torch.uint8, device="cuda")
    sf = torch.full((E * I2 * H // 32,), 0xAA, dtype=torch.uint8, device="cuda")
    B.moe_quantize_weights_fp8(shape, W1, q, sf)
    torch.cuda.synchronize()
    return q, sf


@pytest.mark.parametrize("E,H,I,seed", [(3, 256, 64, 50), (2, 7168, 128, 51), (4, 384, 192, 52)])
def test_quantize_weights_bit_exact(E, H, I, seed):
    g = torch.Generator().manual_seed(seed)
    W1 = (torch.randn(E, H, 2 * I, generator=g) * torch.logspace(-3, 2, 2 * I)).to(torch.bfloat16)
    W1[0, :32, 3] = 0.0  # an all-zero group
    s = B.shape_of(4, H, I, E, 1)
    q, sf = _quantize_w1_gpu(s, W1.cuda())
    rq, rsf = oracle.quantize_weights_fp8(bf16_bits(W1))
    assert np.array_equal(unpack_w1_atoms(sf.cpu().numpy(), E, H, I), rsf), "W1 scales differ from the oracle"
    qg = q.cpu().numpy()
    bad = np.argwhere(qg != rq)
    assert bad.size == 0, f"{len(bad)} E4M3 bytes of W1 differ, first at {bad[0]}"


def _quantize_w2_gpu(shape, W2):
    E, I, H = W2.shape
    q = torch.full((E, H, I), 0xAA, dtype=torch.uint8, device="cuda")
    sf = torch.full((E * H * I // 32,), 0xAA, dtype=torch.uint8, device="cuda")
    B.moe_quantize_w2_fp8(shape, W2, q, sf)
    torch.cuda.synchronize()
    return q, sf


@pytest.mark.parametrize("E,H,I,seed", [(3, 256, 128, 60), (2, 128, 256, 61), (1, 7168, 2048, 62)])
def test_quantize_w2_bit_exact(E, H, I, seed):
    g = torch.Generator().manual_seed(seed)
    W2 = (torch.randn(E, I, H, generator=g) * torch.logspace(-3, 2, H)).to(torch.bfloat16)
    W2[0, :32, 3] = 0.0  # an all-zero group
    s = B.shape_of(4, H, I, E, 1)
    q, sf = _quantize_w2_gpu(s, W2.cuda())
    rq, rsf = oracle.quantize_w2_fp8(bf16_bits(W2))
    assert np.array_equal(unpack_w2_atoms(sf.cpu().numpy(), E, H, I), rsf), "W2 scales differ from the oracle"
    bad = np.argwhere(q.cpu().numpy() != rq)
    assert bad.size == 0, f"{len(bad)} E4M3 bytes of W2 differ, first at {bad[0]}"


def fp8_layer_inputs(T, H, I, E, k, seed):
    """The layer's inputs, quantized on the GPU, and the float64 values the
    E4M3 operands stand for."""
    shape = LayerShape("fp8", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}
    s = B.shape_of(T, H, I, E, k)
    q, sf = _quantize_gpu(s, inp["x"])
    w1q, w1sf = _quantize_w1_gpu(s, inp["W1"])
    w2q, w2sf = _quantize_w2_gpu(s, inp["W2"])
    deq = dict(x=oracle.dequantize_fp8(q.cpu().numpy(), sf.cpu().numpy()),
               W1=dequantized_w1(w1q.cpu().numpy(), w1sf.cpu().numpy(), E, H, I).double().numpy(),
               W2=dequantized_w2(w2q.cpu().numpy(), w2sf.cpu().numpy(), E, H, I).double().numpy())
    return inp, (q, sf, w1q, w1sf, w2q, w2sf), deq


def saved_a8(run, T, I, k):
    """The E4M3 rows of a and their scales from saved's a region
    (include/moe_layer.h, moe_forward_fp8)."""
    L = B.moe_workspace_layout(run.shape)
    R = L.rows_cap
    sv = run.saved.cpu().numpy()
    a8 = sv[L.a: L.a + R * I].reshape(R, I)
    asf = sv[L.a + R * I: L.a + R * I + R * (I // 32)].reshape(R, I // 32)
    return a8, asf


@pytest.mark.parametrize("T,H,I,E,k,seed", [
    (300, 256, 128, 6, 3, 40),    # ragged experts
    (64, 128, 128, 8, 2, 41),     # one K block in each GEMM
    (513, 512, 256, 16, 4, 42),
    (1000, 256, 128, 4, 1, 43),   # ~250 rows per expert: 256-row units (accumulator 0 twice in a row) and 2-chunk experts
    (40, 384, 384, 64, 2, 44),    # experts of 0-5 rows
])
def test_forward_fp8_parity(T, H, I, E, k, seed):
    inp, (q, sf, w1q, w1sf, w2q, w2sf), deq = fp8_layer_inputs(T, H, I, E, k, seed)
    run = GpuRun(T, H, I, E, k)
    run.poison()
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run.route, run.saved, run.y)
    torch.cuda.synchronize()
    ref_tables = oracle_route(inp, E)
    check_tables(run, ref_tables)
    # a second launch on the same tables (its unit feeds must start from the
    # counters the first one left at zero) gives the same bytes
    y2 = torch.full_like(run.y, float("nan"))
    B.moe_forward_fp8(run.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run.route, run.saved, y2)
    torch.cuda.synchronize()
    assert torch.equal(y2, run.y), "a second FP8 forward on the same routing tables differs"
    idx = inp["topk_idx"].cpu().numpy().astype(np.int32)
    w = inp["topk_w"].cpu().numpy()
    y_ref, aq, asf_ref = oracle.forward_fp8(deq["x"], deq["W1"], deq["W2"], idx, w)
    # the quantized activations between the GEMMs
    a8, asf = saved_a8(run, T, I, k)
    perm = ref_tables["perm"]
    _, _, pad = check_a8_against_oracle(a8, asf, perm, aq, asf_ref, k)
    # the L2 GEMM alone, on the GPU's own E4M3 a (exact operands): y from
    # the dequantized rows of a, the dequantized W2 and the weights, in
    # float64, slot by slot
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    a_deq = table[a8] * np.repeat(np.ldexp(1.0, asf.astype(np.int64) - 127), 32, axis=1)
    y_l2 = np.zeros((T, H))
    rows = np.nonzero(perm >= 0)[0]
    for r in rows:
        s_ = perm[r]
        t, j = divmod(int(s_), k)
        y_l2[t] += float(w[t, j]) * (a_deq[r] @ deq["W2"][idx[t, j]])
    compare("y (fp8) vs the L2 contraction of its own E4M3 a", f32(run.y), y_l2)
    compare("y (fp8) vs oracle.forward_fp8", f32(run.y), y_ref)
    # padding rows of the units (inside a 32-row chunk) hold zeros
    written = np.zeros(len(perm), bool)
    offs, counts = ref_tables["offs"], ref_tables["counts"]
    for e in range(E):
        c = int(counts[e])
        if c:
            nsub = (c + 255) // 256
            nb = ((c + nsub - 1) // nsub + 31) // 32 * 32
            for jj in range(nsub):
                lo = offs[e] + jj * nb
                written[lo: lo + ((min(nb, c - jj * nb) + 31) // 32) * 32] = True
    padw = pad[written[pad]]
    assert not a8[padw].any() and np.all(asf[padw] == 127), "padding rows of a are not zero"


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


def test_fp8_experts_wrapper_matches_abi():
    """layer.FP8Experts (weights quantized once, x cast per call) gives the
    bytes of the ABI sequence it marshals, with and without a workspace."""
    from routed_grouped_gemm_routing_gb300.layer import FP8Experts, MoEWorkspace
    T, H, I, E, k = 300, 256, 128, 6, 3
    inp, (q, sf, w1q, w1sf, w2q, w2sf), _ = fp8_layer_inputs(T, H, I, E, k, seed=45)
    run = GpuRun(T, H, I, E, k)
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run.route, run.saved, run.y)
    experts = FP8Experts(inp["W1"], inp["W2"])
    assert torch.equal(experts.W1_fp8, w1q) and torch.equal(experts.W2_sf, w2sf)
    y = experts(inp["x"], inp["topk_idx"].long(), inp["topk_w"])
    ws = MoEWorkspace(T, H, I, E, k)
    y2 = experts(inp["x"], inp["topk_idx"], inp["topk_w"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y, run.y) and torch.equal(y2, run.y)
    with pytest.raises(ValueError):
        FP8Experts(inp["W1"][:, :, :192].contiguous(), inp["W2"][:, :96].contiguous())


def test_fp8_forward_cuda_graph_replay_matches_eager():
    """moe_quantize_fp8 + moe_route_prologue + moe_forward_fp8 captured in a
    CUDA graph (no host synchronisation on the FP8 path) and replayed give
    the eager output bit for bit."""
    T, H, I, E, k = 300, 256, 128, 6, 3
    inp, (q, sf, w1q, w1sf, w2q, w2sf), _ = fp8_layer_inputs(T, H, I, E, k, 70)

    def forward(run, xq, xsf):
        B.moe_quantize_fp8(run.shape, inp["x"], xq, xsf)
        B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
        B.moe_forward_fp8(run.shape, xq, xsf, w1q, w1sf, w2q, w2sf, inp["topk_w"], run.route, run.saved, run.y)

    eager = GpuRun(T, H, I, E, k)
    forward(eager, torch.empty_like(q), torch.empty_like(sf))
    torch.cuda.synchronize()
    run = GpuRun(T, H, I, E, k)
    xq, xsf = torch.empty_like(q), torch.empty_like(sf)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        forward(run, xq, xsf)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    run.poison()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        forward(run, xq, xsf)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(run.y, eager.y)
