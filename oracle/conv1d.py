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
Element types (section "Accuracy Tests" lists fp32 and bf16, and mixed input and state
dtypes): x, weight, bias and out share the input type; the conv state and the window share
the state type; each is bf16 (stored as uint16 bits) or fp32.  The window and state
entries are the row's values stored in the state type: a bf16 value widens to fp32
exactly, an fp32 input narrows to bf16 rounding to nearest, ties to even.  The outputs are
computed from the inputs as given, not from their copies in the state type.
Everything is computed in fp64 from the inputs; results are not rounded here.
"""
from __future__ import annotations

import numpy as np

K = 4
PAD_SLOT = -1


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    bits32 = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return bits32.view(np.float32).astype(np.float64)


def as_f64(a: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) or fp32 values -> fp64."""
    a = np.asarray(a)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Finite fp32 values -> bf16 bits, rounded to nearest with ties to even: add just
    under half of the dropped 16 bits' range, plus the kept part's lowest bit, and
    truncate."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def stored_as(a: np.ndarray, dtype) -> np.ndarray:
    """Values of a (bf16 bits or fp32) as elements of dtype (np.uint16 for bf16 bits, or
    np.float32)."""
    a = np.asarray(a)
    if a.dtype == dtype:
        return a
    if dtype == np.float32:
        return bf16_to_f64(a).astype(np.float32)
    return f32_to_bf16(a)


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
    conv_state after the call, window after the call; both in the state type)."""
    x = np.asarray(c.x)
    state = np.array(c.conv_state, copy=True)
    window = np.array(c.window, copy=True)
    w = as_f64(c.weight)
    bias = None if c.bias is None else as_f64(c.bias)
    out = np.full((c.bs, c.T, c.dim), np.nan)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == PAD_SLOT:
            continue
        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1
        cols = c.conv_state[slot][:, o:o + K - 1]                 # [dim, 3], state type
        xs = x[b].T                                               # [dim, T], input type
        f_bits = np.concatenate([cols, stored_as(xs, cols.dtype)], axis=1)   # row as stored
        out[b] = conv_outputs(np.concatenate([as_f64(cols), as_f64(xs)], axis=1), w, bias,
                              c.silu)
        window[slot] = f_bits[:, 1:]
        state[slot][:, :K - 1] = f_bits[:, c.T:]
    return out, state, window


def per_token_windows(c):
    """The intermediate windows step by step, as the per-token stores write them into a
    dense [bs, T, dim, 3] buffer: window t is the last K - 1 columns of the row after token
    t was appended (in the state type; padded rows left as zeros)."""
    res = np.zeros((c.bs, c.T, c.dim, K - 1), dtype=c.conv_state.dtype)
    for b in range(c.bs):
        slot = int(c.slots[b])
        if slot == PAD_SLOT:
            continue
        o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1
        hist = [c.conv_state[slot][:, o + i] for i in range(K - 1)]
        for t in range(c.T):
            hist.append(stored_as(c.x[b, t], c.conv_state.dtype))
            res[b, t] = np.stack(hist[-(K - 1):], axis=1)
    return res
