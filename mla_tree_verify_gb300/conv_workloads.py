"""Seeded synthetic inputs for the conv-state update of chain speculative verify.

This module only draws inputs; it holds none of the convolution's arithmetic, so both the
CUDA path and the fp64 oracle can use it.

A case is one ``causal_conv1d_update`` call of conv width K = 4 on ``bs`` requests of T
draft tokens each (layouts, all C-contiguous numpy arrays; each floating array is bf16,
stored as uint16 bits, or fp32: x, weight, bias and out in the input type, conv_state and
window in the state type):

* ``x``          ``[bs, T, dim]`` the draft tokens' conv inputs, one row per token.
* ``conv_state`` ``[num_slots, dim, state_len]`` the conv state pool; request b's state
  starts at column ``num_accept[b] - 1`` (0 when there is no accept count) of slot
  ``slots[b]``.
* ``weight``     ``[dim, 4]``, ``bias`` ``[dim]`` (or None).
* ``slots``      int32 ``[bs]``: each request's slot, distinct; -1 marks a padded row.
* ``num_accept`` int32 ``[bs]`` or None.
* ``window``     ``[num_slots, dim, T + 2]`` the deduplicated intermediate-window rows;
  filled with a sentinel so that rows the call must not touch can be checked.
* ``out``        ``[bs, T, dim]`` initial contents (sentinel).

Values: x, state, weight and bias are N(0, 1) (weights scaled by 1/2), rounded to bf16
where the type is bf16; the draws are the same for every choice of types.
"""
from __future__ import annotations

import dataclasses

import numpy as np

K = 4
PAD_SLOT = -1
SENTINEL = np.uint16(0x7F80 | 0x0041)   # a bf16 NaN pattern that no computation produces
SENTINEL_F32 = np.uint32(0x7F800000 | 0x00410041)   # the fp32 one
DTYPES = {"bf16": np.uint16, "f32": np.float32}


def _bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + (0x7FFF + ((u >> 16) & 1))) >> 16).astype(np.uint16)


def _as(a: np.ndarray, dtype: str) -> np.ndarray:
    return _bf16(a) if dtype == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def _filled(shape, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return np.full(shape, SENTINEL, dtype=np.uint16)
    return np.full(shape, SENTINEL_F32, dtype=np.uint32).view(np.float32)


def dtype_name(a: np.ndarray) -> str:
    return "bf16" if a.dtype == np.uint16 else "f32"


@dataclasses.dataclass
class ConvCase:
    x: np.ndarray
    conv_state: np.ndarray
    weight: np.ndarray
    bias: np.ndarray | None
    slots: np.ndarray
    num_accept: np.ndarray | None
    window: np.ndarray
    out: np.ndarray
    silu: bool

    @property
    def bs(self) -> int:
        return self.x.shape[0]

    @property
    def T(self) -> int:
        return self.x.shape[1]

    @property
    def dim(self) -> int:
        return self.x.shape[2]

    @property
    def x_dtype(self) -> str:
        return dtype_name(self.x)

    @property
    def state_dtype(self) -> str:
        return dtype_name(self.conv_state)

    @property
    def num_slots(self) -> int:
        return self.conv_state.shape[0]

    @property
    def state_len(self) -> int:
        return self.conv_state.shape[2]

    def algorithmic_bytes(self) -> int:
        """Bytes a call must move once: x read, out written, per live request the state's
        three read and three written columns and the window row written, and the weights
        and bias read."""
        live = int((self.slots != PAD_SLOT).sum())
        xb, sb = self.x.itemsize, self.conv_state.itemsize
        per_row = self.dim * (xb * (self.T + self.T) + sb * (3 + 3 + (self.T + 2)))
        return live * per_row + self.dim * xb * (K + (1 if self.bias is not None else 0))


def case(seed: int, bs: int, T: int, dim: int, *, num_slots: int | None = None,
         state_len: int = K - 1, accept: bool = False, pad_rows: int = 0,
         bias: bool = True, silu: bool = True, x_dtype: str = "bf16",
         state_dtype: str = "bf16") -> ConvCase:
    """Draws one case.  ``pad_rows`` requests (at random positions) are padded rows;
    ``accept`` draws num_accept[b] in [1, state_len - 2]; ``x_dtype`` (x, weight, bias,
    out) and ``state_dtype`` (conv state, window) are "bf16" or "f32"."""
    if x_dtype not in DTYPES or state_dtype not in DTYPES:
        raise ValueError("dtypes are bf16 or f32")
    if state_len < K - 1:
        raise ValueError("state_len must be at least K - 1")
    num_slots = num_slots or 2 * bs + 3
    if num_slots < bs:
        raise ValueError("fewer slots than requests")
    rng = np.random.default_rng(seed)
    x = _as(rng.standard_normal((bs, T, dim), dtype=np.float32), x_dtype)
    conv_state = _as(rng.standard_normal((num_slots, dim, state_len), dtype=np.float32),
                     state_dtype)
    weight = _as(0.5 * rng.standard_normal((dim, K), dtype=np.float32), x_dtype)
    b_arr = _as(rng.standard_normal(dim, dtype=np.float32), x_dtype) if bias else None
    slots = rng.permutation(num_slots)[:bs].astype(np.int32)
    if pad_rows:
        slots[rng.choice(bs, size=min(pad_rows, bs), replace=False)] = PAD_SLOT
    num_accept = (rng.integers(1, state_len - K + 3, size=bs, endpoint=False).astype(np.int32)
                  if accept else None)
    window = _filled((num_slots, dim, T + K - 2), state_dtype)
    out = _filled((bs, T, dim), x_dtype)
    return ConvCase(x=x, conv_state=conv_state, weight=weight, bias=b_arr, slots=slots,
                    num_accept=num_accept, window=window, out=out, silu=silu)


# The shapes of the GB300 kernel-time table in the pull request "jianc99/sglang#1"
# (deduplicated conv window), section "Benchmarking and Profiling": dim 10240, K 4, bf16.
BENCH_DIM = 10240
BENCH_ROWS = ((1, 8), (64, 8), (128, 8), (128, 16))
