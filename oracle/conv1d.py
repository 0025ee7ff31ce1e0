"""fp64 CPU oracle for the conv-state update of chain speculative verify, with the
intermediate conv window stored deduplicated.

TEST INFRASTRUCTURE ONLY: the tests and bench.py's CPU-baseline leg use it; the product
library never imports it, and it shares no code with the CUDA path.

What it follows: the pull request "jianc99/sglang#1" (deduplicated conv window).
  * section "Motivation": causal_conv1d_update of a chain verify keeps, per draft step,
    the conv window after that step, so that the state of the accepted prefix can be
    restored; the deduplicated layout keeps one [dim, T + K - 2] row per state slot,
    viewed as [T, dim, K - 1] windows whose step stride equals the window stride.
  * section "Modifications": step t's window is columns t .. t + 2 of the row
    [state[1], state[2], x_0, ..., x_{T-1}]; the row is written once; padded rows store
    nothing; the tile applies to conv width 4 only.
  * section "Accuracy Tests": a num_accept_tokens offset into the state.
The convolution itself is the standard causal depthwise one that causal_conv1d_update
names (width K = 4, optional bias and SiLU).  Readings where the page is silent (the
offset's meaning, the state update, the layouts) are the ones in the design notes:
  * request b's state is columns o .. o + 2 of its slot's conv state, o = num_accept - 1
    (0 without accept counts);
  * full row f = [s_0, s_1, s_2, x_0, ..., x_{T-1}];
    out[t] = act(bias + sum_k w[k] f[t + k]);
    window row = f[1 .. T + 2] (so window t = f[t + 1 .. t + 3], the state after step t);
    the state's columns 0 .. 2 become f[T .. T + 2] (the state after the last step).
Everything is computed in fp64 from the bf16 inputs; bf16 results are not rounded here.
"""
from __future__ import annotations

import numpy as np

K = 4
PAD_SLOT = -1


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def full_row(state_cols: np.ndarray, x_tokens: np.ndarray) -> np.ndarray:
    """[dim, 3] state columns and [T, dim] inputs -> [dim, T + 3] row f."""
    return np.concatenate([state_cols, x_tokens.T], axis=1)


def conv_outputs(f: np.ndarray, w: np.ndarray, bias, act: bool) -> np.ndarray:
    """out[t, d] = act(bias[d] + sum_k w[d, k] f[d, t + k]) -> [T, dim]."""
    T = f.shape[1] - (K - 1)
    out = np.zeros((T, f.shape[0]))
    for t in range(T):
        acc = np.zeros(f.shape[0]) if bias is None else bias.copy()
        for k in range(K):
            acc = acc + w[:, k] * f[:, t + k]
        out[t] = silu(acc) if act else acc
    return out


def update(c):
    """One call on a ConvCase.  Returns (out [bs, T, dim] fp64 with NaN on padded rows,
    conv_state after the call (bf16 bits), window after the call (bf16 bits))."""
    x = np.asarray(c.x)
    state = np.array(c.conv_state, copy=True)
    window = np.array(c.window, copy=True)
    w = bf16_to_f64(c.weight)
    bias = None if c.bias is None else bf16_to_f64(c.bias)
    out = np.full((c.bs, c.T, c.dim), np.nan)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == PAD_SLOT:
            continue
        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1
        cols = c.conv_state[slot][:, o:o + K - 1]                 # [dim, 3] bf16 bits
        f_bits = np.concatenate([cols, x[b].T], axis=1)           # [dim, T + 3]
        out[b] = conv_outputs(bf16_to_f64(f_bits), w, bias, c.silu)
        window[slot] = f_bits[:, 1:]
        state[slot][:, :K - 1] = f_bits[:, c.T:]
    return out, state, window


def per_token_windows(c):
    """The intermediate windows step by step, as the per-token stores write them into a
    dense [bs, T, dim, 3] buffer: window t is the last K - 1 columns of the row after token
    t was appended (bf16 bits; padded rows left as zeros)."""
    res = np.zeros((c.bs, c.T, c.dim, K - 1), dtype=np.uint16)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == PAD_SLOT:
            continue
        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1
        hist = [c.conv_state[slot][:, o + i] for i in range(K - 1)]
        for t in range(c.T):
            hist.append(c.x[b, t])
            res[b, t] = np.stack(hist[-(K - 1):], axis=1)
    return res
