"""GPU routing prologue against the oracle's tables, bit for bit, at slot
counts that span one block, many blocks, and blocks of several 1024-slot
rounds; with dropped (-1), out-of-range and duplicate ids, one expert taking
every slot, E = 1 and E = 1024."""
import numpy as np
import pytest
import torch

from moe_testlib import GpuRun, check_tables
import oracle
from routed_grouped_gemm_routing_gb300 import binding as B
from routed_grouped_gemm_routing_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    B.lib()


def _tables(T, E, k, idx: np.ndarray):
    run = GpuRun(T, 64, 64, E, k)
    run.route.fill_(0xFF)
    B.moe_route_prologue(run.shape, torch.as_tensor(idx, dtype=torch.int32).cuda(), run.route)
    torch.cuda.synchronize()
    check_tables(run, oracle.route(idx.astype(np.int32), E, 128))
    return run


def _random_idx(T, E, k, seed, p_drop=0.0, p_bad=0.0):
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, E, size=(T, k), dtype=np.int64)
    u = rng.random((T, k))
    idx[u < p_drop] = -1
    bad = (u >= p_drop) & (u < p_drop + p_bad)
    idx[bad] = rng.choice([E, E + 5, -2, -1000, 2**30], size=int(bad.sum()))
    return idx.astype(np.int32)


@pytest.mark.parametrize("T,E,k,seed", [
    (100, 8, 2, 0),        # less than one round
    (4096, 64, 6, 1),      # 24 blocks of one round, the last one partial
    (8192, 256, 8, 2),     # the V3 routing size: 64 blocks
    (20000, 1024, 5, 3),   # E = 1024
    (3000, 1, 1, 4),       # E = 1
    (5000, 101, 4, 6),     # 8 lanes per expert in the block scan, 808 of them: a partly used warp
    (6000, 600, 7, 7),     # one lane per expert, 600 of the 1024 threads
])
def test_random_ids(T, E, k, seed):
    _tables(T, E, k, _random_idx(T, E, k, seed, p_drop=0.05, p_bad=0.02))


def test_blocks_of_several_rounds():
    """1.12 M slots: 1094 rounds of 1024 slots, so each block holds two
    rounds and the in-block rank carries over between rounds."""
    T, E, k = 140000, 96, 8
    run = _tables(T, E, k, _random_idx(T, E, k, 5, p_drop=0.01, p_bad=0.01))
    assert run.L.route_blocks == 547


def test_one_expert_takes_every_slot():
    T, E, k = 5000, 16, 3
    idx = np.full((T, k), 7, np.int32)
    idx[::97, 1] = -1
    _tables(T, E, k, idx)


def test_duplicates_and_invalid_only():
    T, E, k = 3000, 4, 4
    idx = np.tile(np.array([[2, 2, -1, 9]], np.int32), (T, 1))
    run = _tables(T, E, k, idx)
    assert run.tables()["status"][B.STATUS_N_INVALID] == T
