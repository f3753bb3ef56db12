"""GPU parity of the whole layer through the C ABI against the CPU oracle, on
problems small enough for the oracle to cover every output: routing tables
bit-exact; y, dx, dW1, dW2, d(topk_weights) within the bar of
moe_testlib.compare.  Cases span several M/N tiles, ragged expert groups,
I not a multiple of 128, empty experts, duplicate and dropped slots, invalid
expert ids, one token, no tokens.  Also: run-twice bitwise determinism,
CUDA-graph replay equal to eager, the autograd wrapper equal to the ABI."""
import numpy as np
import pytest
import torch

from moe_testlib import GpuRun, check_tables, compare, f32, oracle_all, oracle_route
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import CONFIGS, LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _inputs(shape: LayerShape, seed=0, mutate=None):
    inp = make_layer_inputs(shape, seed=seed, device="cpu")
    if mutate is not None:
        mutate(inp)
    return {k: v.cuda() for k, v in inp.items()}


def _full_check(shape: LayerShape, inp, report=None):
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    run = GpuRun(T, H, I, E, k)
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    check_tables(run, oracle_route(inp, E))
    ref = oracle_all(inp, E)
    compare("y", f32(run.y), ref["y"], report=report)
    compare("dx", f32(run.dx), ref["dx"], report=report)
    compare("dW1", f32(run.dW1), ref["dW1"], report=report)
    compare("dW2", f32(run.dW2), ref["dW2"], report=report)
    compare("dtopk_w", f32(run.dw), ref["dtopk_w"], bf16_output=False, report=report)
    return run


def test_tiny_config():
    """The small configuration: T=64, H=128, I=64, E=8, top-2, seed 0."""
    shape = CONFIGS["tiny"]
    report = {}
    _full_check(shape, _inputs(shape), report)
    for name, r in report.items():
        print(name, {k: f"{v:.3e}" for k, v in r.items()})


@pytest.mark.parametrize("T,H,I,E,k,seed", [
    (300, 256, 192, 6, 3, 1),     # several M tiles per expert, I % 128 == 64, ragged groups
    (257, 384, 320, 4, 2, 2),     # H spans two 256-column tiles with a tail, I tail
    (129, 128, 128, 2, 1, 3),     # 129 routed rows: a full tile plus one row
    (1, 64, 64, 4, 2, 4),         # one token
    (64, 640, 576, 3, 3, 5),      # every expert in every token (k = E)
])
def test_shapes(T, H, I, E, k, seed):
    shape = LayerShape("case", T=T, H=H, I=I, E=E, k=k)
    _full_check(shape, _inputs(shape, seed))


def test_empty_duplicate_dropped_and_invalid_slots():
    shape = LayerShape("edge", T=200, H=128, I=128, E=16, k=4)

    def mutate(inp):
        g = torch.Generator().manual_seed(11)
        idx = torch.randint(0, 6, (200, 4), generator=g, dtype=torch.int32)  # experts 6..15 empty, duplicates
        idx[5, 1] = -1
        idx[17, 0] = -1
        idx[33, 3] = 17          # out of range: counted, dropped
        idx[40, 2] = -7          # negative other than -1: counted, dropped
        inp["topk_idx"] = idx

    inp = _inputs(shape, 6, mutate)
    run = _full_check(shape, inp)
    assert run.tables()["status"][B.STATUS_N_INVALID] == 2
    assert torch.all(run.dW1[6:] == 0) and torch.all(run.dW2[6:] == 0)
    dw = run.dw.cpu()
    assert dw[5, 1] == 0 and dw[33, 3] == 0 and dw[40, 2] == 0


def test_one_hot_expert_long_k():
    """Every token to expert 0 with weight 1: the variable-K weight gradients
    run over 600 rows (10 K blocks incl. a partial one); other experts empty."""
    shape = LayerShape("hot", T=600, H=256, I=128, E=4, k=1)

    def mutate(inp):
        inp["topk_idx"] = torch.zeros(600, 1, dtype=torch.int32)
        inp["topk_w"] = torch.ones(600, 1, dtype=torch.float32)

    _full_check(shape, _inputs(shape, 7, mutate))


# Expert sizes around the weight-gradient slab.  Mean rows per expert 280:
# the 5-block slab (320 rows): 320 fits, 321 needs a second K chunk of one
# row, 700 needs three chunks (its tiles then go in pairs).  Mean 392: the
# 7-block slab (448 rows): 448 fits, 449 needs two chunks, 1000 three.
SLAB_CASES = {"slab5": [320, 321, 700, 0, 59], "slab7": [448, 449, 1000, 0, 59, 400]}


@pytest.mark.parametrize("main_grad", [False, True])
@pytest.mark.parametrize("case", sorted(SLAB_CASES))
def test_experts_around_the_weight_gradient_slab(case, main_grad):
    """Experts at, one row past, and several chunks past the weight-gradient
    slab's capacity (both slab sizes, chosen by the shape), and one empty
    expert, with H = 320 (the last 256-feature tile half past H) and I = 192
    (two streamed dW1 tiles: one pair; one dW2 tile: a pair's lone tile), the
    workspaces starting as NaN bytes; also through the FP32 main-gradient
    entry point."""
    sizes = SLAB_CASES[case]
    T, H, I, E, k = sum(sizes), 320, 192, len(sizes), 1
    shape = LayerShape("slab_edges", T=T, H=H, I=I, E=E, k=k)

    def mutate(inp):
        g = torch.Generator().manual_seed(12)
        idx = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
        inp["topk_idx"] = idx[torch.randperm(T, generator=g)].view(T, 1)

    inp = _inputs(shape, 13, mutate)
    if not main_grad:
        run = _full_check(shape, inp)
        assert torch.all(run.dW1[3] == 0) and torch.all(run.dW2[3] == 0)
        return
    run = GpuRun(T, H, I, E, k)
    run.poison()
    run.run(inp)
    mg1 = torch.zeros(E, H, 2 * I, device="cuda")
    mg2 = torch.zeros(E, I, H, device="cuda")
    B.moe_backward_main_grad(run.shape, inp["dY"], inp["x"], inp["W1"], inp["W2"], inp["topk_w"], run.route,
                             run.saved, run.bwd, run.dx, mg1, mg2, run.dw)
    torch.cuda.synchronize()
    ref = oracle_all(inp, E)
    compare("main_grad_W1", f32(mg1), ref["dW1"])
    compare("main_grad_W2", f32(mg2), ref["dW2"])
    assert torch.equal(mg1.to(torch.bfloat16), run.dW1) and torch.equal(mg2.to(torch.bfloat16), run.dW2)


def test_skewed_routing_small():
    shape = LayerShape("skew_small", T=512, H=256, I=192, E=32, k=4, skew_c=1.0)
    inp = _inputs(shape, 8)
    counts = np.bincount(inp["topk_idx"].cpu().numpy().ravel(), minlength=32)
    assert counts.max() > 256 and (counts == 0).any()  # long K loop and empty experts both occur
    _full_check(shape, inp)


def test_no_tokens():
    T, H, I, E, k = 0, 128, 64, 4, 2
    run = GpuRun(T, H, I, E, k)
    run.poison()
    inp = dict(x=torch.empty(0, H, dtype=torch.bfloat16, device="cuda"),
               W1=torch.randn(E, H, 2 * I, device="cuda").to(torch.bfloat16),
               W2=torch.randn(E, I, H, device="cuda").to(torch.bfloat16),
               dY=torch.empty(0, H, dtype=torch.bfloat16, device="cuda"),
               topk_idx=torch.empty(0, k, dtype=torch.int32, device="cuda"),
               topk_w=torch.empty(0, k, dtype=torch.float32, device="cuda"))
    run.run(inp)
    torch.cuda.synchronize()
    assert torch.all(run.dW1 == 0) and torch.all(run.dW2 == 0)
    st = run.tables()["status"]
    assert st[B.STATUS_MPAD] == 0 and st[B.STATUS_NUM_TILES] == 0


def test_padding_rows_of_saved_activations_are_zero():
    """Each expert's rows are computed in chunks rounded up to 32 rows; the
    rows from its last routed row up to that 32-row boundary are the zero
    padding that the weight-gradient contraction may read (it stops at the
    16-row step holding the last routed row), so they must be exactly 0 even
    when the buffers start out as NaN."""
    shape = LayerShape("pad", T=100, H=128, I=128, E=4, k=2)
    inp = _inputs(shape, 9)
    run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    tabs = run.tables()
    counts, offs = tabs["counts"], tabs["offs"]
    rows = []
    for e in range(shape.E):
        c = int(counts[e])
        rows += range(int(offs[e]) + c, int(offs[e]) + ((c + 31) // 32) * 32)
    pad = torch.as_tensor(rows, dtype=torch.int64, device="cuda")
    assert pad.numel() > 0
    sv = B.saved_tensors(run.shape, run.saved)
    for name in ("h", "a"):
        assert torch.all(sv[name][pad] == 0), name
    bw = B.backward_tensors(run.shape, run.bwd)
    for name in ("dh", "aw"):
        assert torch.all(bw[name][pad] == 0), name


def test_deterministic_bitwise():
    shape = LayerShape("det", T=300, H=256, I=192, E=6, k=3)
    inp = _inputs(shape, 10)
    outs = []
    for _ in range(2):
        run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
        run.poison()
        run.run(inp)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (run.y, run.dx, run.dW1, run.dW2, run.dw)] + [run.route.clone()])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b)


def test_cuda_graph_replay_matches_eager():
    shape = LayerShape("graph", T=257, H=256, I=128, E=5, k=2)
    inp = _inputs(shape, 11)
    eager = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    eager.run(inp)
    torch.cuda.synchronize()
    run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    run.poison()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run.run(inp, stream=s)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    run.poison()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run.run(inp)
    g.replay()
    torch.cuda.synchronize()
    for a, b in ((run.y, eager.y), (run.dx, eager.dx), (run.dW1, eager.dW1), (run.dW2, eager.dW2),
                 (run.dw, eager.dw)):
        assert torch.equal(a, b)


def test_autograd_wrapper_matches_abi():
    from routed_grouped_gemm_routing_gb300.layer import moe_layer

    shape = LayerShape("ag", T=130, H=128, I=128, E=4, k=2)
    inp = _inputs(shape, 12)
    ref = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    ref.run(inp)
    x = inp["x"].clone().requires_grad_(True)
    W1 = inp["W1"].clone().requires_grad_(True)
    W2 = inp["W2"].clone().requires_grad_(True)
    w = inp["topk_w"].clone().requires_grad_(True)
    y = moe_layer(x, W1, W2, inp["topk_idx"].to(torch.int64), w)
    y.backward(inp["dY"])
    torch.cuda.synchronize()
    assert torch.equal(y, ref.y)
    assert torch.equal(x.grad, ref.dx) and torch.equal(W1.grad, ref.dW1) and torch.equal(W2.grad, ref.dW2)
    assert torch.equal(w.grad, ref.dw)


def test_autograd_workspace_reuse_is_detected():
    """Two forwards on one caller workspace before their backwards: the
    first backward would read the second forward's routing and activations,
    so it raises; the second backward is the layer's gradient (oracle)."""
    from routed_grouped_gemm_routing_gb300.layer import MoEWorkspace, moe_layer

    shape = LayerShape("reuse", T=96, H=128, I=64, E=5, k=2)
    first, second = _inputs(shape, 30), _inputs(shape, 31)
    ws = MoEWorkspace(shape.T, shape.H, shape.I, shape.E, shape.k)
    xs, ys = [], []
    for inp in (first, second):
        x = inp["x"].clone().requires_grad_(True)
        xs.append(x)
        ys.append(moe_layer(x, inp["W1"], inp["W2"], inp["topk_idx"], inp["topk_w"], workspace=ws))
    with pytest.raises(RuntimeError, match="overwritten by a later forward"):
        ys[0].backward(first["dY"])
    ys[1].backward(second["dY"])
    torch.cuda.synchronize()
    ref = oracle_all(second, shape.E)
    compare("y (second forward)", f32(ys[1]), ref["y"])
    compare("dx (second forward)", f32(xs[1].grad), ref["dx"])


def test_host_pipeline_matches_abi():
    """Three steps through HostPipeline (uploads of step n+1 and downloads of
    step n overlapping the kernels, double-buffered device slots) give the
    same bytes as three direct runs on the device."""
    from routed_grouped_gemm_routing_gb300.layer import HostPipeline, MoEWorkspace

    shape = LayerShape("pipe", T=200, H=256, I=128, E=6, k=3)
    batches = [_inputs(shape, 20 + i) for i in range(3)]
    W1, W2 = batches[0]["W1"], batches[0]["W2"]
    refs = []
    for inp in batches:
        inp = dict(inp, W1=W1, W2=W2)
        run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
        run.run(inp)
        torch.cuda.synchronize()
        refs.append((run.y.cpu(), run.dx.cpu(), run.dw.cpu(), run.dW1.clone(), run.dW2.clone()))
    ws = MoEWorkspace(shape.T, shape.H, shape.I, shape.E, shape.k)
    pipe = HostPipeline(ws, W1, W2)
    hosts, outs = [], []
    for inp in batches:
        h = {n: inp[n].cpu().pin_memory() for n in ("x", "topk_idx", "topk_w", "dY")}
        o = (torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory(),
             torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory(),
             torch.empty(shape.T, shape.k, dtype=torch.float32).pin_memory())
        hosts.append(h)
        outs.append(o)
        pipe.submit(h["x"], h["topk_idx"], h["topk_w"], h["dY"], *o)
    pipe.synchronize()
    torch.cuda.synchronize()
    for (y, dx, dw), (ry, rdx, rdw, _, _) in zip(outs, refs):
        assert torch.equal(y, ry) and torch.equal(dx, rdx) and torch.equal(dw, rdw)
    assert torch.equal(pipe.dW1, refs[-1][3]) and torch.equal(pipe.dW2, refs[-1][4])
