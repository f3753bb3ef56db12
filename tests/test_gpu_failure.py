"""Failure detection on the GPU without a fault: every mbarrier wait of the
GEMM kernels is bounded, and a wait that runs out raises the kernel's abort
flag, lets the other roles leave their waits, and sets bit 0 of
MOE_STATUS_FLAGS for the host.  moe_selftest_wait_timeout runs the same wait
helpers on a barrier that nothing arrives on, with a 1 ms limit instead of
the kernels' 2 s, so the give-up path itself is exercised: it must end
promptly, report through the status words, and leave the context usable."""
import time

import pytest
import torch

from moe_testlib import GpuRun, compare, f32, oracle_all
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build
from routed_grouped_gemm_routing_gb300.workloads import CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    shape = CONFIGS["tiny"]
    inp = {k: v.cuda() for k, v in make_layer_inputs(shape, seed=0, device="cpu").items()}
    run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    run.run(inp)
    torch.cuda.synchronize()
    assert B.moe_read_status(run.shape, run.route)[B.STATUS_FLAGS] == 0
    y_before = run.y.clone()

    limit_ns = 1_000_000
    elapsed = torch.full((3,), -2, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    B.moe_selftest_wait_timeout(run.shape, run.route, limit_ns, elapsed)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    status = B.moe_read_status(run.shape, run.route)
    el = elapsed.cpu().tolist()
    print("bounded-wait self-test: waits ended after", el, "ns; wall", wall, "s; flags", status[B.STATUS_FLAGS])
    assert status[B.STATUS_FLAGS] & 1, "the timeout was not reported in MOE_STATUS_FLAGS"
    assert limit_ns <= el[0] < 50 * limit_ns, "the timed-out wait did not give up at its limit"
    # the other two wait forms left on the abort flag, before their own 4 ms limit
    assert 0 <= el[1] < 3 * limit_ns and 0 <= el[2] < 3 * limit_ns
    assert wall < 5.0

    # the context still works, and the next prologue clears the flag
    run.poison()
    run.run(inp)
    torch.cuda.synchronize()
    assert B.moe_read_status(run.shape, run.route)[B.STATUS_FLAGS] == 0
    assert torch.equal(run.y, y_before)
    compare("y after the self-test", f32(run.y), oracle_all(inp, shape.E)["y"])


def test_selftest_rejects_limits_out_of_range():
    shape = CONFIGS["tiny"]
    run = GpuRun(shape.T, shape.H, shape.I, shape.E, shape.k)
    for bad in (0, 999, 100_000_001):
        with pytest.raises(B.MoeError):
            B.moe_selftest_wait_timeout(run.shape, run.route, bad)
