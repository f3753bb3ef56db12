"""Pins of the oracle's router top-k (logits -> topk_idx, topk_weights).

Each check compares the oracle with something that is not the oracle: a
library routine (numpy's stable argsort, scipy's softmax), the seeded
workload generator's torch routing, closed forms for constructed rows (ties,
constant shifts, infinities), or a brute-force ordering property.
"""
import numpy as np
import pytest
import torch

import oracle
from routed_grouped_gemm_routing_gb300.workloads import make_routing



def _key(lg):
    k = lg.astype(np.float64).copy()
    k[np.isnan(k)] = -np.inf
    return k


@pytest.mark.parametrize("T,E,k,seed", [(64, 8, 2, 0), (33, 37, 5, 1), (16, 256, 8, 2), (5, 6, 6, 3)])
def test_matches_stable_argsort_and_softmax(T, E, k, seed):
    scipy_special = pytest.importorskip("scipy.special")  # only this pin needs scipy
    lg = np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)
    idx, w = oracle.router_topk(lg, k)
    key = _key(lg)
    want = np.argsort(-key, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, want)
    sel = np.take_along_axis(key, want, axis=1)
    np.testing.assert_allclose(w, scipy_special.softmax(sel, axis=1), rtol=2e-7, atol=1e-9)


def test_matches_workload_generator_routing():
    """The seeded workloads route with torch (stable descending sort, softmax
    over the selected logits in FP32): same ids, weights within FP32 error."""
    T, E, k = 128, 64, 6
    g = torch.Generator()
    g.manual_seed(0 * 7919 + 11)
    logits = torch.randn(T, E, generator=g, dtype=torch.float32)
    want_idx, want_w = make_routing(T, E, k, seed=0)
    idx, w = oracle.router_topk(logits.numpy(), k)
    assert np.array_equal(idx, want_idx.numpy())
    np.testing.assert_allclose(w, want_w.numpy(), rtol=2e-6, atol=1e-7)


def test_ties_go_to_the_lower_expert_id():
    lg = np.zeros((3, 9), np.float32)
    lg[1, [2, 5, 7]] = 1.0  # three equal maxima
    lg[2, :] = -3.5
    idx, w = oracle.router_topk(lg, 4)
    assert idx[0].tolist() == [0, 1, 2, 3] and np.allclose(w[0], 0.25)
    assert idx[1].tolist() == [2, 5, 7, 0]
    e = np.exp(-1.0)
    np.testing.assert_allclose(w[1], np.array([1, 1, 1, e]) / (3 + e), rtol=1e-7)
    assert idx[2].tolist() == [0, 1, 2, 3] and np.allclose(w[2], 0.25)


def test_signed_zeros_are_equal_keys():
    """-0 and +0 are the same number: their order comes from the expert id."""
    lg = np.full((2, 6), -1.0, np.float32)
    lg[0, [1, 4]] = [0.0, -0.0]
    lg[1, [1, 4]] = [-0.0, 0.0]
    idx, w = oracle.router_topk(lg, 3)
    assert idx[0].tolist() == [1, 4, 0] and idx[1].tolist() == [1, 4, 0]
    np.testing.assert_allclose(w[0], np.array([1, 1, np.exp(-1.0)]) / (2 + np.exp(-1.0)), rtol=1e-7)


def test_shift_invariance():
    lg = np.random.default_rng(5).standard_normal((20, 12)).astype(np.float32)
    i0, w0 = oracle.router_topk(lg, 3)
    i1, w1 = oracle.router_topk(lg + np.float32(64.0), 3)
    assert np.array_equal(i0, i1)
    np.testing.assert_allclose(w0, w1, rtol=1e-5)


def test_k_equals_e_is_a_full_softmax():
    lg = np.random.default_rng(6).standard_normal((7, 10)).astype(np.float32)
    idx, w = oracle.router_topk(lg, 10)
    assert all(sorted(r) == list(range(10)) for r in idx.tolist())
    z = lg.astype(np.float64)
    full = np.exp(z - z.max(axis=1, keepdims=True))  # FP64 softmax written out with numpy
    full /= full.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx, axis=1), rtol=2e-7)


def test_nan_and_infinities():
    nan, inf = np.float32("nan"), np.float32("inf")
    lg = np.array([
        [nan, 0.5, nan, -1.0, 2.0],     # NaN ranks below every number
        [1.0, inf, 3.0, inf, 0.0],      # two +inf: 1/2 each, 0 elsewhere
        [-inf, -inf, -inf, -inf, -inf],  # all -inf: uniform
        [nan, nan, nan, nan, nan],      # all NaN = all -inf
    ], np.float32)
    idx, w = oracle.router_topk(lg, 3)
    assert idx[0].tolist() == [4, 1, 3]
    assert idx[1].tolist() == [1, 3, 2] and w[1].tolist() == [0.5, 0.5, 0.0]
    assert idx[2].tolist() == [0, 1, 2] and np.allclose(w[2], 1 / 3)
    assert idx[3].tolist() == [0, 1, 2] and np.allclose(w[3], 1 / 3)
    # a row with one NaN among the selected after the numbers run out
    idx2, w2 = oracle.router_topk(np.array([[nan, 1.0, nan]], np.float32), 2)
    assert idx2[0].tolist() == [1, 0] and w2[0].tolist() == [1.0, 0.0]


def test_selection_property_brute_force():
    """Every selected key beats every unselected one (a tie only with a higher
    id), and the selected list is in decreasing key order: checked pair by
    pair on small rows with many repeated values."""
    rng = np.random.default_rng(7)
    lg = rng.integers(-3, 4, size=(200, 7)).astype(np.float32)
    for k in (1, 3, 7):
        idx, _ = oracle.router_topk(lg, k)
        for t in range(lg.shape[0]):
            sel = idx[t].tolist()
            assert len(set(sel)) == k
            for a, b in zip(sel, sel[1:]):
                assert lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
            for e in set(range(7)) - set(sel):
                for s in sel:
                    assert lg[t, s] > lg[t, e] or (lg[t, s] == lg[t, e] and s < e)
