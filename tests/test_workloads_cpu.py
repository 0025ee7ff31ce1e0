"""The seeded input generator's slot layouts: every layout references distinct, in-range
slots, holds the same rows (so the attention result does not depend on the layout), and
'contiguous' / 'runs' really place rows in consecutive slots."""
import numpy as np
import pytest


from mla_tree_verify_gb300 import workloads as W



def _slots(wl):
    out = []
    for b in range(wl.bs):
        out.append(wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]].astype(np.int64))
        out.append(wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]])
    return np.concatenate(out)


@pytest.mark.parametrize("layout", ["scattered", "contiguous", "runs"])
def test_layout_slots_and_rows(layout):
    P, T = [300, 1000, 0, 129], [5, 16, 3, 1]
    base = W.build("t", 11, P, T, "random", 30000)
    wl = W.build("t", 11, P, T, "random", 30000, layout=layout)
    s, s0 = _slots(wl), _slots(base)
    assert len(np.unique(s)) == len(s) and s.min() >= 0 and s.max() < wl.num_slots
    # the row at every referenced position is the same as in the scattered layout
    assert np.array_equal(wl.kv_cache[s], base.kv_cache[s0])
    assert np.array_equal(wl.q, base.q) and np.array_equal(wl.custom_mask, base.custom_mask)
    # every other slot is poisoned
    rest = np.setdiff1d(np.arange(wl.num_slots), s)
    assert (wl.kv_cache[rest] == W.BF16_NAN).all()
    step = np.diff(s)
    if layout == "contiguous":
        assert (step == 1).all()
    elif layout == "runs":
        assert (step == 1).mean() > 0.95 and (step != 1).any()


def test_unknown_layout_rejected():
    with pytest.raises(ValueError):
        W.build("t", 1, [10], [2], "chain", 100, layout="striped")
