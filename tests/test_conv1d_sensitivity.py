"""The conv-update oracle's pins are sensitive: each planted mistake makes at least one of
them fail.

Each case loads a copy of oracle/conv1d.py with one plausible mistake (an off-by-one in
the window or the state, a dropped accept offset, reversed taps, a dropped bias, the
activation in the wrong place, padded rows computed, outputs taken from the row as stored
in the state type, fp32 to bf16 narrowing that truncates or rounds ties away from zero, the
window left in the input type) and runs the pins of
tests/test_conv1d_cpu.py against it on the CPU.  The unmodified source passes all of them.
"""
import importlib.util
import os

import pytest

import test_conv1d_cpu as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "conv1d.py")

MUTATIONS = {
    "none": None,
    "window_starts_one_column_early": ("window[slot] = f_bits[:, 1:]",
                                       "window[slot] = f_bits[:, :-1]"),
    "state_keeps_one_column_too_early": ("state[slot][:, :K - 1] = f_bits[:, c.T:]",
                                         "state[slot][:, :K - 1] = f_bits[:, c.T - 1:-1]"),
    "accept_offset_ignored": ("o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1\n"
                              "        cols",
                              "o = 0\n        cols"),
    "taps_reversed": ("acc = acc + w[:, k] * f[:, t + k]", "acc = acc + w[:, K - 1 - k] * f[:, t + k]"),
    "bias_dropped": ("acc = np.zeros(f.shape[0]) if bias is None else bias.copy()",
                     "acc = np.zeros(f.shape[0])"),
    "activation_before_bias": ("out[t] = silu(acc) if act else acc",
                               "out[t] = (silu(acc - (0 if bias is None else bias)) + "
                               "(0 if bias is None else bias)) if act else acc"),
    "padded_rows_computed": ("        if slot == PAD_SLOT:\n            continue\n"
                             "        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1\n"
                             "        cols",
                             "        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1\n"
                             "        cols"),
    "outputs_from_the_stored_row": ("out[b] = conv_outputs(np.concatenate([as_f64(cols), "
                                    "as_f64(xs)], axis=1), w, bias,",
                                    "out[b] = conv_outputs(as_f64(f_bits), w, bias,"),
    "narrowing_truncates": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)",
                            "return (u >> 16).astype(np.uint16)"),
    "narrowing_ties_away_from_zero": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16)"
                                      ".astype(np.uint16)",
                                      "return ((u + 0x8000) >> 16).astype(np.uint16)"),
    "window_keeps_the_input_type": ("f_bits = np.concatenate([cols, stored_as(xs, cols.dtype)], "
                                    "axis=1)",
                                    "f_bits = np.concatenate([cols, xs], axis=1)"),
}

PINS = [pins.test_hand_derived_case, pins.test_two_calls_equal_one_call, pins.test_copy_taps,
        pins.test_silu_applied_to_the_biased_sum,
        pins.test_padded_rows_and_other_slots_untouched, pins.test_accept_offset_changes_the_state_read,
        lambda: pins.test_window_row_is_the_per_token_windows(8, True, 12),
        pins.test_bf16_narrowing_hand_values, pins.test_mixed_types_outputs_use_the_inputs_as_given,
        pins.test_mixed_types_bf16_inputs_fp32_state]


def _variant(name, tmp_path):
    src = open(SRC).read()
    mut = MUTATIONS[name]
    if mut is not None:
        old, new = mut
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    path = os.path.join(tmp_path, f"conv1d_{name}.py")
    with open(path, "w") as f:
        f.write(src)
    spec = importlib.util.spec_from_file_location(f"conv1d_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_the_mutation(name, tmp_path, monkeypatch):
    mod = _variant(name, tmp_path)
    monkeypatch.setattr(pins, "O", mod)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, TypeError):
            failures += 1
    if name == "none":
        assert failures == 0
    else:
        assert failures > 0, f"no pin catches {name}"
