"""GPU parity of the router top-k entry point (moe_router_topk) against the
CPU oracle: topk_idx and the routing tables bit-exact, topk_w within FP32
rounding of the oracle's FP64 softmax (|err| <= 2e-6 * w + 1e-7, the error
of an FP32 exp, sum and division over k <= 1024 terms).  Cases: E not a
multiple of 32, k = 1, k = E, k > 32, ties, NaN and infinite logits, no
tokens, the V3 router shape, run-twice determinism."""
import numpy as np
import pytest
import torch

import oracle
from moe_testlib import check_tables
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


class _Tables:
    """Just what check_tables reads from a GpuRun."""

    def __init__(self, shape, route):
        self.shape, self.route = shape, route

    def tables(self):
        return {k_: v.cpu().numpy() for k_, v in B.route_tables(self.shape, self.route).items()}


def _run(logits: np.ndarray, k: int):
    T, E = logits.shape
    shape = B.shape_of(T, 64, 64, E, k)
    L = B.moe_workspace_layout(shape)
    route = torch.full((max(L.route_bytes, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    lg = torch.as_tensor(logits, device="cuda")
    idx = torch.full((max(T, 1), k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((max(T, 1), k), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_router_topk(shape, lg, idx, w, route)
    torch.cuda.synchronize()
    return shape, route, idx[:T].cpu().numpy(), w[:T].cpu().numpy()


def _check(logits: np.ndarray, k: int):
    shape, route, idx, w = _run(logits, k)
    ref_idx, ref_w = oracle.router_topk(logits, k)
    assert np.array_equal(idx, ref_idx), "topk_idx differs from the oracle"
    assert np.all(np.abs(w - ref_w) <= 2e-6 * np.abs(ref_w) + 1e-7), float(np.max(np.abs(w - ref_w)))
    check_tables(_Tables(shape, route), oracle.route(ref_idx, logits.shape[1], 128))


@pytest.mark.parametrize("T,E,k,seed", [
    (300, 64, 6, 0), (257, 37, 5, 1), (64, 7, 7, 2), (100, 1024, 1, 3), (40, 200, 33, 4), (9, 1024, 1024, 5),
    (130, 100, 4, 6), (50, 500, 9, 7), (33, 32, 32, 8), (70, 33, 3, 9), (60, 993, 17, 10),
])
def test_random_logits(T, E, k, seed):
    rng = np.random.default_rng(seed)
    _check((rng.standard_normal((T, E)) * 2).astype(np.float32), k)


def test_ties_nan_and_infinities():
    rng = np.random.default_rng(8)
    lg = rng.integers(-2, 3, size=(120, 45)).astype(np.float32)  # many equal logits
    lg[3, :] = np.nan
    lg[4, :] = -np.inf
    lg[5, [1, 7, 30]] = np.inf
    lg[6, ::3] = np.nan
    lg[7, 10] = np.inf
    lg[8, :] = -1.0
    lg[8, [3, 20]] = [0.0, -0.0]      # equal keys: +0 at the lower id
    lg[9, :] = -1.0
    lg[9, [2, 40]] = [-0.0, 0.0]      # equal keys: -0 at the lower id
    lg[10, ::2] = -0.0                # -0 and (integer-valued) others
    _check(lg, 4)
    _check(lg, 45)


def test_v3_router_shape():
    g = torch.Generator()
    g.manual_seed(11)
    _check(torch.randn(8192, 256, generator=g, dtype=torch.float32).numpy(), 8)


def test_no_tokens():
    shape, route, idx, w = _run(np.zeros((0, 16), np.float32), 2)
    st = B.route_tables(shape, route)["status"].cpu().numpy()
    assert st[B.STATUS_MPAD] == 0 and st[B.STATUS_NUM_TILES] == 0


def test_deterministic():
    lg = np.random.default_rng(9).standard_normal((2000, 256)).astype(np.float32)
    _, _, i1, w1 = _run(lg, 8)
    _, _, i2, w2 = _run(lg, 8)
    assert np.array_equal(i1, i2) and np.array_equal(w1.view(np.int32), w2.view(np.int32))


def test_cuda_graph_replay_matches_eager():
    """The router and the routing prologue captured in a CUDA graph (no host
    synchronisation inside moe_router_topk) and replayed give the eager
    results bit for bit, routing tables included."""
    lg = torch.as_tensor(np.random.default_rng(21).standard_normal((3000, 64)).astype(np.float32), device="cuda")
    T, E, k = 3000, 64, 6
    shape = B.shape_of(T, 64, 64, E, k)
    L = B.moe_workspace_layout(shape)

    def bufs():
        return (torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
                torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((max(L.route_bytes, 16),), 0xFF, dtype=torch.uint8, device="cuda"))

    idx_e, w_e, route_e = bufs()
    B.moe_router_topk(shape, lg, idx_e, w_e, route_e)
    idx_g, w_g, route_g = bufs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.moe_router_topk(shape, lg, idx_g, w_g, route_g)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    idx_g.fill_(-7)
    w_g.fill_(float("nan"))
    route_g.fill_(0xFF)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.moe_router_topk(shape, lg, idx_g, w_g, route_g)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(idx_g, idx_e)
    assert torch.equal(w_g.view(torch.int32), w_e.view(torch.int32))
    assert torch.equal(route_g, route_e)
