"""Pins for the oracle's routing tables (DeepGEMM Mega-MoE article, "Block-M
Alignment for Irregular Token Counts"; Primus-Turbo Mega MoE README,
"Implementation Map": dispatch prologue builds routing tables).

The tables are pinned by a hand-worked example and by invariants that
together determine them uniquely (counts, block-M padded offsets, every
expert's rows holding exactly its slots in increasing slot order, padding
rows = -1, inverse permutation, tile owner table)."""
import numpy as np
import pytest

import oracle


def test_hand_worked_example():
    # T=3 tokens, k=2, E=3 experts, block M = 4.
    # slots s = t*k + j:  s0->e2  s1->e0  s2->e0  s3->e2  s4->e1  s5->e0
    # counts = [3, 1, 2]; each pads to 4 rows -> offs = [0, 4, 8, 12]
    # expert 0 rows 0..3 hold slots 1, 2, 5 then a pad row
    # expert 1 rows 4..7 hold slot 4 then 3 pad rows
    # expert 2 rows 8..11 hold slots 0, 3 then 2 pad rows
    idx = np.array([[2, 0], [0, 2], [1, 0]], np.int32)
    r = oracle.route(idx, E=3, bm=4)
    assert r["counts"].tolist() == [3, 1, 2]
    assert r["offs"].tolist() == [0, 4, 8, 12]
    assert r["perm"].tolist() == [1, 2, 5, -1, 4, -1, -1, -1, 0, 3, -1, -1]
    assert r["inv"].tolist() == [8, 0, 1, 9, 4, 2]
    assert r["tiles"].tolist() == [0, 1, 2]
    assert (r["mpad"], r["num_tiles"], r["n_invalid"]) == (12, 3, 0)
    # capacity bound: floor((6 + 3*3) / 4) * 4 = 12
    assert oracle.rows_cap(3, 3, 2, 4) == 12


def _check_invariants(idx, E, bm, r):
    T, k = idx.shape
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E)
    assert np.array_equal(r["counts"], counts)
    assert r["n_invalid"] == int(np.sum(~valid & (flat != -1)))
    offs = r["offs"]
    assert offs[0] == 0
    sizes = np.diff(offs)
    assert np.all(sizes % bm == 0)
    assert np.all(sizes >= counts) and np.all(sizes - counts < bm)  # smallest multiple of bm
    assert r["mpad"] == offs[-1] and r["num_tiles"] * bm == r["mpad"]
    cap = oracle.rows_cap(T, E, k, bm)
    assert len(r["perm"]) == cap and r["mpad"] <= cap and cap % bm == 0
    perm, inv = r["perm"], r["inv"]
    for e in range(E):
        rows = perm[offs[e]: offs[e + 1]]
        held = rows[: counts[e]]
        assert np.array_equal(held, np.nonzero(flat == e)[0]), "rows must hold the expert's slots in slot order"
        assert np.all(rows[counts[e]:] == -1)
    assert np.all(perm[r["mpad"]:] == -1)
    for s in range(T * k):
        if valid[s]:
            assert perm[inv[s]] == s
        else:
            assert inv[s] == -1
    tiles = r["tiles"]
    for m in range(len(tiles)):
        if m < r["num_tiles"]:
            e = tiles[m]
            assert offs[e] <= m * bm < offs[e + 1]
        else:
            assert tiles[m] == -1


@pytest.mark.parametrize("T,E,k,bm,seed", [(64, 8, 2, 128, 0), (37, 5, 3, 4, 1), (200, 16, 4, 8, 2),
                                           (1, 4, 4, 128, 3), (50, 64, 6, 16, 4)])
def test_invariants_random(T, E, k, bm, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _check_invariants(idx, E, bm, oracle.route(idx, E, bm))


def test_duplicates_dropped_invalid_and_empty_experts():
    rng = np.random.default_rng(5)
    T, E, k, bm = 40, 9, 3, 4
    idx = rng.integers(0, 4, size=(T, k)).astype(np.int32)  # experts 4..8 empty, duplicates allowed
    idx[3, 1] = -1
    idx[7, 0] = -1
    idx[9, 2] = 11      # out of range: counted and dropped
    idx[10, 0] = -5     # negative other than -1: counted and dropped
    r = oracle.route(idx, E, bm)
    _check_invariants(idx, E, bm, r)
    assert r["n_invalid"] == 2
    assert np.all(r["counts"][4:] == 0)


def test_worst_case_capacity_is_reached():
    # every expert gets exactly one slot: each pads to a full block
    T, E, k, bm = 8, 8, 1, 128
    idx = np.arange(T, dtype=np.int32).reshape(T, 1)
    r = oracle.route(idx, E, bm)
    assert r["mpad"] == E * bm == oracle.rows_cap(T, E, k, bm)
    _check_invariants(idx, E, bm, r)


def test_no_tokens():
    idx = np.zeros((0, 2), np.int32)
    r = oracle.route(idx, 4, 128)
    assert r["mpad"] == 0 and r["num_tiles"] == 0 and len(r["perm"]) == 0
    assert r["counts"].tolist() == [0, 0, 0, 0] and r["offs"].tolist() == [0] * 5
