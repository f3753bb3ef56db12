"""The allocation-free inference forward, moe_forward_noalloc.

It serves callers that cannot allocate device memory when they run the
layer (a plugin inside an inference engine that is given no workspace, a
serving loop that must not call cudaMalloc because it can synchronise the
device): routing tables and intermediates live in a static device array
inside the library.  Checked through the C ABI against the workspace-based
moe_route_prologue + moe_forward (bit for bit: same kernels, same order) and
against the CPU oracle with the tolerance of every other parity test, on two
calls in a row (the second with other routing and another shape, so stale
scratch contents would show); its status words are read back; a shape whose
scratch need sits just under the static array's size runs, one just over it
is rejected.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import GpuRun, compare, f32
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import LayerShape, bf16_bits, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _scratch_need(T, H, I, E, k):
    L = B.moe_workspace_layout(B.shape_of(T, H, I, E, k))
    return ((L.route_bytes + 255) // 256) * 256 + L.saved_bytes


def _forward_both(shape, seed, mutate=None):
    inp = make_layer_inputs(shape, seed=seed, device="cpu", with_grad_out=False)
    if mutate is not None:
        mutate(inp)
    inp = {k: v.cuda() for k, v in inp.items()}
    ref = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    ref.run(inp, backward=False)
    y = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.full((B.STATUS_WORDS,), -7, dtype=torch.int32, device="cuda")
    B.moe_forward_noalloc(B.shape_of(shape.T, shape.H, shape.I, shape.E, shape.k), inp["x"], inp["W1"], inp["W2"],
                          inp["topk_idx"], inp["topk_w"], y, status_out=status)
    torch.cuda.synchronize()
    return inp, y, ref, status.cpu().numpy()


def _oracle_forward(inp):
    return oracle.forward(bf16_bits(inp["x"]), bf16_bits(inp["W1"]), bf16_bits(inp["W2"]),
                          inp["topk_idx"].cpu().numpy().astype(np.int32),
                          inp["topk_w"].cpu().numpy().astype(np.float32))


def _check(shape, inp, y, ref, status):
    assert torch.equal(y, ref.y)  # same kernels, same order: identical bits
    compare(f"y ({shape.name}) vs oracle", f32(y), _oracle_forward(inp))
    want = B.moe_read_status(ref.shape, ref.route)
    for w in (B.STATUS_MPAD, B.STATUS_NUM_TILES, B.STATUS_N_INVALID, B.STATUS_FLAGS, B.STATUS_NUM_PAIRS):
        assert status[w] == want[w], (w, status[w], want[w])
    assert status[B.STATUS_FLAGS] == 0


def test_noalloc_forward_matches_workspace_forward_twice():
    first = LayerShape("noalloc_a", T=64, H=128, I=64, E=8, k=2)
    second = LayerShape("noalloc_b", T=150, H=256, I=192, E=6, k=3)

    def invalid_ids(inp):  # two out-of-range ids and one dropped slot: counted and skipped
        inp["topk_idx"][3, 1] = 99
        inp["topk_idx"][10, 0] = -5
        inp["topk_idx"][11, 2] = -1

    for shape, seed, mutate in ((first, 0, None), (second, 1, invalid_ids)):
        inp, y, ref, status = _forward_both(shape, seed, mutate)
        _check(shape, inp, y, ref, status)
        if mutate is not None:
            assert status[B.STATUS_N_INVALID] == 2


def test_noalloc_at_the_scratch_limit():
    """The largest hidden size whose scratch need fits the static array runs
    (bit-equal to the workspace path, within the bar of the oracle); 64 more
    is rejected before any launch."""
    T, I, E, k = 64, 64, 8, 2
    H = 64
    while _scratch_need(T, H + 64, I, E, k) <= B.NOALLOC_SCRATCH_BYTES:
        H += 64
    assert B.NOALLOC_SCRATCH_BYTES - _scratch_need(T, H, I, E, k) < 64 * 1024 * 4
    shape = LayerShape("noalloc_limit", T=T, H=H, I=I, E=E, k=k)
    inp, y, ref, status = _forward_both(shape, 2)
    _check(shape, inp, y, ref, status)

    over = B.shape_of(T, H + 64, I, E, k)
    assert _scratch_need(T, H + 64, I, E, k) > B.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    fn = B.lib().moe_forward_noalloc
    fn.argtypes = [B.ctypes.POINTER(B.MoeShape)] + [B.ctypes.c_void_p] * 8
    fn.restype = B.ctypes.c_int
    p = dummy.data_ptr()
    assert fn(B.ctypes.byref(over), p, p, p, p, p, p, None, None) == B.MOE_EUNSUPPORTED
    assert "static scratch" in B.moe_last_error()


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    s = B.shape_of(4096, 2048, 1408, 64, 6)  # needs ~410 MB of scratch
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    fn = B.lib().moe_forward_noalloc
    fn.argtypes = [B.ctypes.POINTER(B.MoeShape)] + [B.ctypes.c_void_p] * 8
    fn.restype = B.ctypes.c_int
    p = dummy.data_ptr()
    assert fn(B.ctypes.byref(s), p, p, p, p, p, p, None, None) == B.MOE_EUNSUPPORTED  # rejected before any launch
    assert "static scratch" in B.moe_last_error()
