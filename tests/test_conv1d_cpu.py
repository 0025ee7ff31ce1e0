"""Pins of the conv-state update oracle (chain verify, deduplicated conv window, K = 4).

The oracle is checked against a hand-derived case, against the per-token definition of the
intermediate windows (read through the overlapping [T, dim, 3] view of the deduplicated
row), against splitting a call's tokens over two calls, and against taps that reduce the
convolution to a copy.
"""
import json
import os

import numpy as np
import pytest

import oracle.conv1d as O
from mla_tree_verify_gb300 import conv_workloads as CW

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(a):
    return CW._bf16(np.asarray(a, dtype=np.float32))


def _golden():
    g = json.load(open(os.path.join(HERE, "golden", "conv1d_case.json")))
    c = CW.ConvCase(x=_bits(g["x"]), conv_state=_bits(g["conv_state"]), weight=_bits(g["weight"]),
                    bias=_bits(g["bias"]), slots=np.array(g["slots"], np.int32),
                    num_accept=np.array(g["num_accept"], np.int32),
                    window=np.full((2, g["dim"], g["T"] + 2), CW.SENTINEL, np.uint16),
                    out=np.full((3, g["T"], g["dim"]), CW.SENTINEL, np.uint16), silu=g["silu"])
    return g, c


def test_hand_derived_case():
    g, c = _golden()
    out, state, window = O.update(c)
    for b, exp in enumerate(g["expect_out"]):
        if exp is None:
            assert np.isnan(out[b]).all()
        else:
            np.testing.assert_array_equal(out[b], np.array(exp))
    np.testing.assert_array_equal(O.bf16_to_f64(window), np.array(g["expect_window"], float))
    np.testing.assert_array_equal(O.bf16_to_f64(state), np.array(g["expect_state"], float))


@pytest.mark.parametrize("T,accept,state_len", [(1, False, 3), (2, True, 5), (3, False, 3),
                                                 (8, True, 12), (9, False, 3), (16, True, 4)])
def test_window_row_is_the_per_token_windows(T, accept, state_len):
    """Reading the deduplicated row through the overlapping view (step stride == window
    stride) gives, for every step, the window that the per-token path writes."""
    c = CW.case(7 + T, bs=5, T=T, dim=24, state_len=state_len, accept=accept, pad_rows=1)
    _, _, window = O.update(c)
    dense = O.per_token_windows(c)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == CW.PAD_SLOT:
            continue
        row = window[slot]                                   # [dim, T + 2]
        view = np.lib.stride_tricks.as_strided(
            row, shape=(T, c.dim, 3), strides=(row.strides[1], row.strides[0], row.strides[1]))
        np.testing.assert_array_equal(view, dense[b])


def test_two_calls_equal_one_call():
    """Feeding T1 tokens then T2 tokens leaves the same state, and gives the same outputs,
    as feeding the T1 + T2 tokens at once (state columns 0..2, no accept offset)."""
    c = CW.case(21, bs=4, T=7, dim=16, silu=False)
    out, state, _ = O.update(c)
    c1 = CW.case(21, bs=4, T=7, dim=16, silu=False)
    c1.x = np.ascontiguousarray(c.x[:, :3])
    c1.window = np.zeros((c.num_slots, c.dim, 5), np.uint16)
    out1, state1, _ = O.update(c1)
    c2 = CW.case(21, bs=4, T=7, dim=16, silu=False)
    c2.conv_state = state1
    c2.x = np.ascontiguousarray(c.x[:, 3:])
    c2.window = np.zeros((c.num_slots, c.dim, 6), np.uint16)
    out2, state2, _ = O.update(c2)
    np.testing.assert_array_equal(np.concatenate([out1, out2], axis=1), out)
    np.testing.assert_array_equal(state2, state)


def test_copy_taps():
    """w = (0, 0, 0, 1) and no bias or activation copy the inputs; w = (1, 0, 0, 0) reads
    the row three columns back."""
    c = CW.case(5, bs=3, T=6, dim=8, bias=False, silu=False)
    c.weight = _bits(np.tile([0, 0, 0, 1], (8, 1)))
    out, _, _ = O.update(c)
    np.testing.assert_array_equal(out, O.bf16_to_f64(c.x))
    c.weight = _bits(np.tile([1, 0, 0, 0], (8, 1)))
    out, _, window = O.update(c)
    for b in range(3):
        f = np.concatenate([c.conv_state[c.slots[b]][:, :3], c.x[b].T], axis=1)
        np.testing.assert_array_equal(out[b], O.bf16_to_f64(f[:, :6]).T)


def test_silu_closed_forms():
    v = np.array([-30.0, -1.0, 0.0, 1.0, 30.0])
    s = O.silu(v)
    assert s[2] == 0.0
    np.testing.assert_allclose(s - O.silu(-v), v, rtol=0, atol=1e-12)     # silu(v) - silu(-v) = v
    np.testing.assert_allclose(s[3], 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    assert abs(s[4] - 30.0) < 1e-11 and abs(s[0]) < 1e-11


def test_padded_rows_and_other_slots_untouched():
    c = CW.case(9, bs=6, T=4, dim=12, pad_rows=2, num_slots=20)
    out, state, window = O.update(c)
    live = set(int(s) for s in c.slots if s != CW.PAD_SLOT)
    for s in range(c.num_slots):
        if s not in live:
            assert (window[s] == CW.SENTINEL).all()
            np.testing.assert_array_equal(state[s], c.conv_state[s])
    for b in range(c.bs):
        assert np.isnan(out[b]).all() == (c.slots[b] == CW.PAD_SLOT)


def test_accept_offset_changes_the_state_read():
    """With state_len 5 the accept count selects which three columns start the row."""
    c = CW.case(3, bs=2, T=2, dim=4, state_len=5, accept=True, silu=False)
    for n in (1, 2, 3):
        c.num_accept = np.array([n, n], np.int32)
        _, _, window = O.update(c)
        s = c.slots[0]
        np.testing.assert_array_equal(window[s][:, :2], c.conv_state[s][:, n:n + 2])


def test_silu_applied_to_the_biased_sum():
    """With copy taps and a bias beta, out(x) - out(-x - 2 beta) = x + beta exactly when the
    activation is applied to the whole biased sum (silu(v) - silu(-v) = v).  x and beta
    are multiples of 1/8, so -x - 2 beta is exact in bf16."""
    rng = np.random.default_rng(12)
    c = CW.case(11, bs=2, T=4, dim=8, silu=True)
    c.weight = _bits(np.tile([0, 0, 0, 1], (8, 1)))
    beta = rng.integers(-12, 13, size=8) / 8.0
    xs = rng.integers(-24, 25, size=(2, 4, 8)) / 8.0
    c.bias = _bits(beta)
    c.x = _bits(xs)
    c2 = CW.case(11, bs=2, T=4, dim=8, silu=True)
    c2.weight, c2.bias = c.weight, c.bias
    c2.x = _bits(-xs - 2 * beta)
    assert np.array_equal(O.bf16_to_f64(c2.x), -xs - 2 * beta)
    out1, _, _ = O.update(c)
    out2, _, _ = O.update(c2)
    np.testing.assert_allclose(out1 - out2, xs + beta, rtol=0, atol=1e-12)
