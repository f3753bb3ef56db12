"""The expected scheduling tables of the SM-pair GEMMs (pair_offs,
pair_owner; include/moe_layer.h) on a hand-worked example, so that the
helper the GPU parity tests compare the prologue's tables with is itself
pinned."""
import numpy as np

from moe_testlib import walk_tables


def test_walk_tables_hand_example():
    # counts 3, 300, 0, 300, 129 -> block-128 padded sizes 128, 384, 0, 384, 256
    # -> tile pairs 1, 2, 0, 2, 1; walk by decreasing count, ties by id:
    # e1 (300), e3 (300), e4 (129), e0 (3), e2 (0)
    counts = [3, 300, 0, 300, 129]
    offs = np.concatenate([[0], np.cumsum([128, 384, 0, 384, 256])])
    pair_offs, owner = walk_tables(counts, offs, 9)
    assert pair_offs.tolist() == [5, 0, 6, 2, 4, 6]
    assert owner.tolist() == [1, 1, 3, 3, 4, 0, -1, -1, -1]
