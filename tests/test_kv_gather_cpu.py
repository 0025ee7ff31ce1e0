"""Pins of the oracle's KV gather-copy (no GPU).

The gather is its own definition (dst[j] = kv[kv_indices[kv_indptr[0] + j]], zero rows
for out-of-pool slots, new index dst_slot0 + j), so it is pinned against a hand-derived
case, a scatter back to the source slots, and its argument checks.
"""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_hand_derived_case():
    case = json.load(open(os.path.join(HERE, "golden", "kv_gather_case.json")))
    kv = np.zeros((case["num_slots"], 576), dtype=np.uint16)
    for s in range(case["num_slots"]):
        kv[s, :] = 0x4000 + s
    dst, new, bad = oracle.kv_gather(kv, case["kv_indices"], case["kv_indptr"],
                                     case["dst_rows"], case["dst_slot0"])
    for j, bits in enumerate(case["expected_row_bits"]):
        assert (dst[j] == bits).all()
    assert new.tolist() == case["expected_new_indices"]
    assert bad == case["expected_bad"]


def test_scatter_back_restores_the_referenced_rows():
    rng = np.random.default_rng(5)
    kv = rng.integers(0, 1 << 16, size=(300, 576), dtype=np.uint16)
    idx = rng.permutation(300)[:120].astype(np.int32)
    ptr = np.array([0, 17, 17, 80, 120], dtype=np.int32)
    dst, new, bad = oracle.kv_gather(kv, idx, ptr, 128, 1000)
    assert bad == 0
    back = np.zeros_like(kv)
    back[idx] = dst[:120]
    assert (back[idx] == kv[idx]).all()
    assert (new == 1000 + np.arange(120)).all()
    assert (dst[120:] == 0).all()          # rows past the batch are not written


def test_indices_offset_by_the_first_indptr():
    # kv_indptr[0] > 0: entry i lands at row i - kv_indptr[0]
    kv = np.zeros((8, 576), dtype=np.uint16)
    for s in range(8):
        kv[s] = s + 1
    idx = np.array([9, 9, 3, 1, 7], dtype=np.int32)     # entries 0, 1 are not in the batch
    dst, new, bad = oracle.kv_gather(kv, idx, [2, 4, 5], 3, 50)
    assert [int(dst[j, 0]) for j in range(3)] == [4, 2, 8]
    assert new[2:].tolist() == [50, 51, 52] and bad == 0


def test_bad_arguments():
    kv = np.zeros((4, 576), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_gather(kv, [0, 1, 2], [0, 2, 1], 3, 0)      # decreasing indptr
    with pytest.raises(ValueError):
        oracle.kv_gather(kv, [0, 1, 2], [0, 3], 2, 0)         # too few destination rows
    dst, new, bad = oracle.kv_gather(kv, [0], [0, 0, 0], 1, 0)  # empty batch
    assert bad == 0 and (dst == 0).all()
