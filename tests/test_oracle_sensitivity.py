"""The oracle pins are sensitive: each planted mistake makes at least one of them fail.

Each case copies mla_oracle.c, applies one plausible mistake (a wrong index, a
dropped term, a wrong sign), builds the copy with gcc into a temporary directory
and runs a compact set of pins against it on the CPU.  The unmodified source passes
all of them.
"""
import math
import os
import subprocess

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from mla_tree_verify_gb300 import workloads as W

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "mla_oracle.c")

MUTATIONS = {
    "none": None,
    "mask_row_stride_uses_prefix_len": (
        "in->mask_indptr[b] + i * (P + T) + c", "in->mask_indptr[b] + i * P + c"),
    "values_read_from_rope_offset": (
        "o[d] += p * bf16_value(v[d]);", "o[d] += p * bf16_value(v[d + 64]);"),
    "sm_scale_dropped": ("return in->sm_scale * acc;", "return acc;"),
    "score_skips_rope_dims": ("for (int d = 0; d < D_QK; ++d) acc +=",
                              "for (int d = 0; d < D_V; ++d) acc +="),
    "combine_weight_sign_flipped": ("double w = exp(m[s] - M);", "double w = exp(M - m[s]);"),
    "lse_without_log": ("*lse = M + log(sum);", "*lse = M + sum;"),
    "draft_slot_off_by_one": ("in->out_cache_loc[in->qo_indptr[b] + (c - P)]",
                              "in->out_cache_loc[in->qo_indptr[b] + (c - P + 1) % (T_ + 0)]"),
}


def _build_variant(tmp_path, name):
    src = open(SRC).read()
    mut = MUTATIONS[name]
    if mut is not None:
        old, new = mut
        assert old in src, old
        src = src.replace(old, new)
        if "T_" in new:  # the off-by-one needs the draft count in scope
            src = src.replace("  int64_t slot;\n  if (c < P)",
                              "  int64_t slot;\n  int64_t T_ = in->qo_indptr[b + 1] - in->qo_indptr[b];"
                              "\n  if (c < P)")
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    so = os.path.join(tmp_path, f"lib_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", so, path, "-lm"],
                   check=True)
    return oracle.load_library(so)


def _f(bits):
    return W.bf16_bits_to_float32(bits).astype(np.float64)


def _pin_dense_tree(lib):
    """Masked softmax written with numpy on a random-tree workload."""
    wl = W.build("s", 7, [13, 6], [4, 5], "random", 80, heads=2)
    out, lse = oracle.Oracle(wl, lib=lib).attend()
    out = out.reshape(wl.total_q, wl.num_heads, W.D_V)
    lse = lse.reshape(wl.total_q, wl.num_heads)
    q, kv = _f(wl.q), _f(wl.kv_cache)
    for b in range(wl.bs):
        rows = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]],
                               wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]])
        K = kv[rows]
        Q = q[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]
        S = wl.sm_scale * np.einsum("thd,ld->thl", Q, K)
        vis = wl.mask_block(b).astype(bool)
        S = np.where(vis[:, None, :], S, -np.inf)
        ref = np.einsum("thl,lv->thv", softmax(S, axis=-1), K[:, :W.D_V])
        sl = slice(int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1]))
        if not (np.allclose(out[sl], ref, rtol=1e-10, atol=1e-12)
                and np.allclose(lse[sl], logsumexp(S, axis=-1), rtol=1e-10, atol=1e-12)):
            return False
    return True


def _pin_split(lib):
    wl = W.build("s", 8, [40], [3], "random", 90, heads=1)
    orc = oracle.Oracle(wl, lib=lib)
    full, full_lse = orc.attend()
    cuts = [0, 5, 17, 30, 43]
    for r in range(wl.total_q):
        parts = [orc.partial(r, 0, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        out, lse = oracle.combine([p[0] for p in parts], [p[1] for p in parts],
                                  np.stack([p[2] for p in parts]), lib=lib)
        if not (np.allclose(out, full[r], rtol=1e-12, atol=1e-13)
                and abs(lse - full_lse[r]) < 1e-12 * (1 + abs(lse))):
            return False
    return True


def _pin_single_key(lib):
    wl = W.build("s", 9, [0], [3], "chain", 10, heads=1)
    wl.custom_mask[:] = np.eye(3, dtype=np.uint8).reshape(-1)
    out, lse = oracle.Oracle(wl, lib=lib).attend()
    kv, q = _f(wl.kv_cache), _f(wl.q)
    for r in range(3):
        s = int(wl.out_cache_loc[r])
        if not np.array_equal(out[r], kv[s, :W.D_V]):
            return False
        if abs(lse[r] - wl.sm_scale * float(q[r, 0] @ kv[s])) > 1e-12:
            return False
    return True


PINS = [_pin_dense_tree, _pin_split, _pin_single_key]


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build_variant(str(tmp_path), name)
    results = [pin(lib) for pin in PINS]
    if name == "none":
        assert all(results), results
    else:
        assert not all(results), f"mistake {name} passed every pin"
