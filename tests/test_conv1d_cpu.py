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


# Element types.  The pull request "jianc99/sglang#1", section "Accuracy Tests", lists fp32
# and bf16, and mixed input and state dtypes.  The window and state hold the row's values in
# the state type; the outputs are computed from the inputs as given.

def test_bf16_narrowing_hand_values():
    """Round to nearest, ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 and goes
    to the even one (1); 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 and
    goes up; anything above halfway goes up; negatives mirror; fp32's largest value lies
    above halfway between bf16's largest, (2 - 2^-7) 2^127, and 2^128, so it overflows."""
    v = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20, 1 + 2**-8 - 2**-20,
                  -(1 + 3 * 2**-8), 0.0, -0.0, np.finfo(np.float32).max], np.float32)
    got = O.f32_to_bf16(v)
    exp = np.array([0x3F80, 0x3F82, 0x3F81, 0x3F80, 0xBF82, 0x0000, 0x8000, 0x7F80], np.uint16)
    np.testing.assert_array_equal(got, exp)


def test_bf16_narrowing_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormals
                        np.ldexp(rng.integers(1 << 23, 1 << 24, 2000), -23 - 7).astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(O.f32_to_bf16(v), ref)


def test_widening_is_exact():
    bits = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]                    # finite values only
    wide = O.stored_as(bits, np.float32)
    assert wide.dtype == np.float32
    np.testing.assert_array_equal(O.f32_to_bf16(wide), bits)
    np.testing.assert_array_equal(wide.astype(np.float64), O.bf16_to_f64(bits))


def _widen(c):
    """The same case with every bf16 array widened to fp32 (exact)."""
    import dataclasses
    f = lambda a: None if a is None else (O.stored_as(a, np.float32) if a.dtype == np.uint16 else a)
    return dataclasses.replace(c, x=f(c.x), conv_state=f(c.conv_state), weight=f(c.weight),
                               bias=f(c.bias), window=f(c.window), out=f(c.out))


@pytest.mark.parametrize("T,accept", [(1, False), (8, True), (16, True)])
def test_fp32_of_bf16_values_equals_bf16(T, accept):
    """fp32 inputs that hold bf16 values give the bf16 call's results, widened."""
    c = CW.case(40 + T, bs=4, T=T, dim=24, state_len=6, accept=accept, pad_rows=1)
    out, state, window = O.update(c)
    out32, state32, window32 = O.update(_widen(c))
    assert state32.dtype == np.float32 and window32.dtype == np.float32
    np.testing.assert_array_equal(out32, out)
    np.testing.assert_array_equal(state32, O.stored_as(state, np.float32))
    live = [int(s) for s in c.slots if s != CW.PAD_SLOT]
    np.testing.assert_array_equal(window32[live], O.stored_as(window[live], np.float32))


def test_mixed_types_outputs_use_the_inputs_as_given():
    """fp32 inputs, bf16 state, copy taps (out[t] = x_t): the outputs are the fp32 inputs
    exactly, while the window and state hold them rounded to bf16."""
    c = CW.case(50, bs=3, T=5, dim=16, bias=False, silu=False, x_dtype="f32")
    c.weight = np.zeros_like(c.weight)
    c.weight[:, 3] = 1.0
    out, state, window = O.update(c)
    assert window.dtype == np.uint16 and state.dtype == np.uint16
    for b in range(c.bs):
        s = int(c.slots[b])
        np.testing.assert_array_equal(out[b], c.x[b].astype(np.float64))
        assert not np.array_equal(out[b], O.bf16_to_f64(O.f32_to_bf16(c.x[b])))
        np.testing.assert_array_equal(window[s][:, 2:], O.f32_to_bf16(c.x[b]).T)
        np.testing.assert_array_equal(state[s][:, :3], O.f32_to_bf16(c.x[b][2:]).T)


def test_mixed_types_bf16_inputs_fp32_state():
    """bf16 inputs, fp32 state: the window's input columns are the inputs widened, its first
    two columns the state's values unchanged."""
    c = CW.case(51, bs=3, T=4, dim=16, state_len=5, accept=True, state_dtype="f32")
    _, state, window = O.update(c)
    for b in range(c.bs):
        s, o = int(c.slots[b]), int(c.num_accept[b]) - 1
        np.testing.assert_array_equal(window[s][:, 2:], O.bf16_to_f64(c.x[b]).T.astype(np.float32))
        np.testing.assert_array_equal(window[s][:, :2], c.conv_state[s][:, o + 1:o + 3])
        np.testing.assert_array_equal(state[s][:, 3:], c.conv_state[s][:, 3:])


@pytest.mark.parametrize("xd,sd", [("f32", "bf16"), ("bf16", "f32"), ("f32", "f32")])
def test_window_row_is_the_per_token_windows_mixed(xd, sd):
    c = CW.case(60, bs=4, T=7, dim=24, state_len=5, accept=True, pad_rows=1, x_dtype=xd,
                state_dtype=sd)
    _, _, window = O.update(c)
    dense = O.per_token_windows(c)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == CW.PAD_SLOT:
            continue
        for t in range(c.T):
            np.testing.assert_array_equal(window[slot][:, t:t + 3], dense[b, t])
