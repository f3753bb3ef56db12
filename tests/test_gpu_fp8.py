"""GPU parity of the FP8 path through the C ABI.

* moe_quantize_fp8 and moe_quantize_weights_fp8: E4M3 bytes and UE8M0 scale
  bytes bit-exact against the oracle's quantization (integer output: exact
  bar; the weights' scales read back from the kernel's atom layout);
* moe_forward_fp8 (block-scaled tensor-core MMA on the E4M3 operands): y
  within the comparison bar of the oracle's forward on the dequantized input
  and dequantized W1, and of moe_forward run on them in bf16 (every product
  of two E4M3 values and two powers of two is exact in FP32, so the two
  differ only in how the MMAs round FP32 partial sums: bit for bit on these
  small shapes, one bf16 step in a few elements at the V3 shape);
* moe_dequantize_fp8 bit-exact against the oracle's dequantization."""
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


def unpack_w1_atoms(atoms, E, H, I):
    """The weights' scale bytes [E, 2I, H // 32] from the kernel's atom layout
    (include/moe_layer.h, moe_quantize_weights_fp8)."""
    a = np.asarray(atoms).reshape(E, I // 64, H // 128, 512)
    f = np.arange(2 * I)
    fi = np.where(f < I, f, f - I)
    g, r = fi // 64, np.where(f < I, 0, 64) + fi % 64
    out = np.zeros((E, 2 * I, H // 32), np.uint8)
    for j32 in range(H // 32):
        out[:, :, j32] = a[:, g, j32 // 4, 16 * (r % 32) + 4 * (r // 32) + j32 % 4]
    return out


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


def dequantized_w1(q, sf_atoms, E, H, I):
    """bf16 W1 [E, H, 2I] from its E4M3 bytes (K-major) and scale atoms (exact)."""
    deq = oracle.dequantize_fp8(np.asarray(q).reshape(E * 2 * I, H),
                                unpack_w1_atoms(sf_atoms, E, H, I).reshape(E * 2 * I, H // 32))
    return torch.from_numpy(np.ascontiguousarray(deq.reshape(E, 2 * I, H).transpose(0, 2, 1)).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("T,H,I,E,k,seed", [
    (300, 256, 192, 6, 3, 40),    # ragged experts, I % 128 == 64
    (64, 128, 64, 8, 2, 41),      # one K block
    (513, 512, 256, 16, 4, 42),
    (1000, 256, 128, 4, 1, 43),   # ~250 rows per expert: 256-row units (accumulator 0 twice in a row) and 2-chunk experts
])
def test_forward_fp8_parity(T, H, I, E, k, seed):
    shape = LayerShape("fp8", T=T, H=H, I=I, E=E, k=k)
    inp = {n: v.cuda() for n, v in make_layer_inputs(shape, seed=seed, device="cpu").items()}
    s = B.shape_of(T, H, I, E, k)
    q, sf = _quantize_gpu(s, inp["x"])
    wq, wsf = _quantize_w1_gpu(s, inp["W1"])
    xd = _dequantized_bf16(q.cpu().numpy(), sf.cpu().numpy()).cuda()
    W1d = dequantized_w1(wq.cpu().numpy(), wsf.cpu().numpy(), E, H, I).cuda()
    # the bf16 path on the dequantized operands
    ref_run = GpuRun(T, H, I, E, k)
    ref_run.run(dict(inp, x=xd, W1=W1d), backward=False)
    # the FP8 path
    run = GpuRun(T, H, I, E, k)
    run.poison()
    B.moe_route_prologue(run.shape, inp["topk_idx"], run.route)
    B.moe_forward_fp8(run.shape, q, sf, wq, wsf, inp["W2"], inp["topk_w"], run.route, run.saved, run.y)
    torch.cuda.synchronize()
    check_tables(run, oracle_route(inp, E))
    # a second launch on the same tables (its unit feed must start from the
    # counters the first one left at zero) gives the same bytes
    y2 = torch.full_like(run.y, float("nan"))
    B.moe_forward_fp8(run.shape, q, sf, wq, wsf, inp["W2"], inp["topk_w"], run.route, run.saved, y2)
    torch.cuda.synchronize()
    assert torch.equal(y2, run.y), "a second FP8 forward on the same routing tables differs"
    # every E4M3 x E4M3 x 2^k product is exact in FP32; the two MMA kinds may
    # still round their FP32 partial sums differently over a long K
    compare("y (fp8) vs bf16 path on the dequantized operands", f32(run.y), f32(ref_run.y))
    print("fp8 forward equal to the bf16 path bit for bit:", bool(torch.equal(run.y, ref_run.y)))
    y_ref = oracle.forward(bf16_bits(xd.cpu()), bf16_bits(W1d.cpu()), bf16_bits(inp["W2"].cpu()),
                           inp["topk_idx"].cpu().numpy().astype(np.int32), inp["topk_w"].cpu().numpy())
    compare("y (fp8) vs oracle on the dequantized operands", f32(run.y), y_ref)
    # the quantization error of the input stays within E4M3's half step
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
