"""Pins for the fp64 oracle: checks against things other than the oracle itself.

No source page prints a worked example of the attention, so every pin comes from the
mathematics of masked softmax attention (brute force, closed forms, textbook dense
attention, invariances) and from the hand-derived cases in tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from mla_tree_verify_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(bits):
    return W.bf16_bits_to_float32(bits).astype(np.float64)


def small(seed, P, T, tree="random", heads=4, pool=None, **kw):
    pool = pool or (sum(P) + sum(T) + 7) * 2
    return W.build("small", seed, P, T, tree, pool, heads=heads, **kw)


# ---------------------------------------------------------------------------
# 1. Brute force on tiny inputs: softmax written out with no max subtraction,
#    exact sums (math.fsum), indices read straight from the flat arrays.
# ---------------------------------------------------------------------------
def brute_force(wl, scale):
    q = f32(wl.q)
    kv = f32(wl.kv_cache)
    out = np.zeros((wl.total_q, wl.num_heads, W.D_V))
    lse = np.zeros((wl.total_q, wl.num_heads))
    for b in range(wl.bs):
        P = int(wl.kv_indptr[b + 1]) - int(wl.kv_indptr[b])
        T = int(wl.qo_indptr[b + 1]) - int(wl.qo_indptr[b])
        L = P + T
        keys = [int(wl.kv_indices[int(wl.kv_indptr[b]) + c]) for c in range(P)]
        keys += [int(wl.out_cache_loc[int(wl.qo_indptr[b]) + j]) for j in range(T)]
        for i in range(T):
            r = int(wl.qo_indptr[b]) + i
            vis = [True] * P + [bool(wl.custom_mask[int(wl.mask_indptr[b]) + i * L + P + j])
                                for j in range(T)]
            for h in range(wl.num_heads):
                ws = []
                for c in range(L):
                    if vis[c]:
                        s = scale * math.fsum(q[r, h, d] * kv[keys[c], d] for d in range(W.D_QK))
                        ws.append((math.exp(s), keys[c]))
                Z = math.fsum(w for w, _ in ws)
                for d in range(W.D_V):
                    out[r, h, d] = math.fsum(w * kv[k, d] for w, k in ws) / Z
                lse[r, h] = math.log(Z)
    return out.reshape(-1, W.D_V), lse.reshape(-1)


@pytest.mark.parametrize("seed,P,T,tree", [
    (1, [5], [3], "random"),
    (2, [0, 4], [2, 3], "random"),
    (3, [3, 1], [1, 3], "chain"),
    (4, [2], [3], "random"),
])
def test_brute_force_tiny(seed, P, T, tree):
    wl = small(seed, P, T, tree, heads=2)
    out, lse = oracle.Oracle(wl).attend()
    bo, bl = brute_force(wl, wl.sm_scale)
    np.testing.assert_allclose(out, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, bl, rtol=1e-12, atol=1e-13)


def test_brute_force_random_mask_bits():
    """A mask that is not a tree (random bits, diagonal kept) still matches."""
    wl = small(11, [4, 2], [3, 3], "random", heads=2)
    rng = np.random.default_rng(5)
    for b in range(wl.bs):
        blk = wl.mask_block(b)
        P = int(wl.prefix_lens[b])
        d = blk[:, P:]
        d[...] = rng.integers(0, 2, size=d.shape)
        np.fill_diagonal(d, 1)
    out, lse = oracle.Oracle(wl).attend()
    bo, bl = brute_force(wl, wl.sm_scale)
    np.testing.assert_allclose(out, bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, bl, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# 2. A single visible key returns that key's V row, and lse = its score.
# ---------------------------------------------------------------------------
def test_single_visible_key():
    wl = small(21, [0, 0], [4, 2], "random", heads=3)
    for b in range(wl.bs):  # only the diagonal stays visible
        blk = wl.mask_block(b)
        blk[...] = 0
        np.fill_diagonal(blk, 1)
    out, lse = oracle.Oracle(wl).attend()
    q = f32(wl.q)
    kv = f32(wl.kv_cache)
    k = 0
    for r in range(wl.total_q):
        slot = int(wl.out_cache_loc[r])
        for h in range(wl.num_heads):
            np.testing.assert_array_equal(out[k], kv[slot, :W.D_V])
            s = wl.sm_scale * float(np.dot(q[r, h], kv[slot]))
            assert abs(lse[k] - s) <= 1e-12 * (1 + abs(s))
            k += 1


# ---------------------------------------------------------------------------
# 3. All-visible mask == textbook softmax(Q K^T * scale) V on contiguous rows.
# ---------------------------------------------------------------------------
def test_all_visible_equals_dense():
    wl = small(31, [37, 9], [5, 4], "random", heads=4)
    wl.custom_mask[:] = 1
    out, lse = oracle.Oracle(wl).attend()
    out = out.reshape(wl.total_q, wl.num_heads, W.D_V)
    lse = lse.reshape(wl.total_q, wl.num_heads)
    q = f32(wl.q)
    kv = f32(wl.kv_cache)
    for b in range(wl.bs):
        rows = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]],
                               wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]])
        K = kv[rows]                      # [L, 576]
        V = K[:, :W.D_V]                  # [L, 512]
        Q = q[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]  # [T, H, 576]
        S = wl.sm_scale * np.einsum("thd,ld->thl", Q, K)
        ref = np.einsum("thl,lv->thv", softmax(S, axis=-1), V)
        np.testing.assert_allclose(out[wl.qo_indptr[b]:wl.qo_indptr[b + 1]], ref, rtol=1e-11,
                                   atol=1e-12)
        np.testing.assert_allclose(lse[wl.qo_indptr[b]:wl.qo_indptr[b + 1]],
                                   logsumexp(S, axis=-1), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# 4. Split invariance: partials over any chunking, merged, equal the unsplit result.
#    This also pins the LSE-weighted combine.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("nsplit", [1, 2, 7, 64, "random"])
def test_split_invariance(nsplit):
    wl = small(41, [150, 33], [6, 5], "random", heads=2)
    orc = oracle.Oracle(wl)
    full, full_lse = orc.attend()
    rng = np.random.default_rng(3)
    k = 0
    for b in range(wl.bs):
        L = int(wl.prefix_lens[b] + wl.draft_lens[b])
        if nsplit == "random":
            cuts = np.unique(np.concatenate([[0, L], rng.integers(0, L, size=9)]))
        else:
            chunk = -(-L // nsplit)
            cuts = np.unique(np.minimum(np.arange(nsplit + 1) * chunk, L))
        for i in range(int(wl.draft_lens[b])):
            r = int(wl.qo_indptr[b]) + i
            for h in range(wl.num_heads):
                parts = [orc.partial(r, h, int(c0), int(c1)) for c0, c1 in zip(cuts[:-1], cuts[1:])]
                m = np.array([p[0] for p in parts])
                l = np.array([p[1] for p in parts])
                o = np.stack([p[2] for p in parts])
                out, lse = oracle.combine(m, l, o)
                k = r * wl.num_heads + h
                np.testing.assert_allclose(out, full[k], rtol=1e-12, atol=1e-13)
                assert abs(lse - full_lse[k]) <= 1e-12 * (1 + abs(lse))
                # the same merge written with numpy: weights e^{m_s - M}
                keep = l > 0
                M = m[keep].max()
                w = np.exp(m[keep] - M)
                np.testing.assert_allclose((w[:, None] * o[keep]).sum(0) / (w * l[keep]).sum(),
                                           full[k], rtol=1e-12, atol=1e-13)


def test_combine_skips_empty_partials():
    o = np.random.default_rng(0).standard_normal((3, W.D_V))
    m = np.array([1.5, -np.inf, 0.25])
    l = np.array([2.0, 0.0, 3.0])
    o[1] = np.nan  # an empty split's payload is never read
    out, lse = oracle.combine(m, l, o)
    w = np.exp(np.array([1.5, 0.25]) - 1.5)
    np.testing.assert_allclose(out, (w[0] * o[0] + w[1] * o[2]) / (2.0 * w[0] + 3.0 * w[1]),
                               rtol=1e-14)
    assert abs(lse - (1.5 + math.log(2.0 * w[0] + 3.0 * w[1]))) < 1e-14
    out, lse = oracle.combine(np.array([-np.inf]), np.array([0.0]), np.zeros((1, W.D_V)))
    assert lse == -np.inf and not out.any()


# ---------------------------------------------------------------------------
# 5. A chain mask is causal attention over prefix + drafts.
# ---------------------------------------------------------------------------
def test_chain_equals_causal():
    wl = small(51, [20, 7], [6, 3], "chain", heads=3)
    out, lse = oracle.Oracle(wl).attend()
    out = out.reshape(wl.total_q, wl.num_heads, W.D_V)
    q = f32(wl.q)
    kv = f32(wl.kv_cache)
    for b in range(wl.bs):
        P, T = int(wl.prefix_lens[b]), int(wl.draft_lens[b])
        rows = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]],
                               wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]])
        K = kv[rows]
        Q = q[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]
        S = wl.sm_scale * np.einsum("thd,ld->thl", Q, K)
        causal = np.arange(P + T)[None, :] <= (P + np.arange(T))[:, None]   # [T, L]
        S = np.where(causal[:, None, :], S, -np.inf)
        ref = np.einsum("thl,lv->thv", softmax(S, axis=-1), K[:, :W.D_V])
        np.testing.assert_allclose(out[wl.qo_indptr[b]:wl.qo_indptr[b + 1]], ref, rtol=1e-11,
                                   atol=1e-12)


# ---------------------------------------------------------------------------
# 6. Invariances and special cases.
# ---------------------------------------------------------------------------
def test_slot_permutation_invariance():
    wl = small(61, [30, 12], [4, 5], "random", heads=2, pool=200)
    out, lse = oracle.Oracle(wl).attend()
    perm = np.random.default_rng(9).permutation(wl.num_slots)   # new slot of old slot s
    kv2 = np.empty_like(wl.kv_cache)
    kv2[perm] = wl.kv_cache
    wl.kv_cache = kv2
    wl.kv_indices = perm[wl.kv_indices].astype(np.int32)
    wl.out_cache_loc = perm[wl.out_cache_loc].astype(np.int64)
    out2, lse2 = oracle.Oracle(wl).attend()
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_heads_are_independent():
    wl = small(71, [25], [4], "random", heads=4)
    out, lse = oracle.Oracle(wl).attend()
    wl.q[:, 2, :] = W._bf16_bits(np.random.default_rng(1).standard_normal((wl.total_q, W.D_QK),
                                                                           dtype=np.float32))
    out2, lse2 = oracle.Oracle(wl).attend()
    o = out.reshape(wl.total_q, 4, -1)
    o2 = out2.reshape(wl.total_q, 4, -1)
    for h in (0, 1, 3):
        np.testing.assert_array_equal(o[:, h], o2[:, h])
    assert not np.array_equal(o[:, 2], o2[:, 2])


def test_zero_scale_is_mean_of_visible_rows():
    wl = small(81, [9, 0], [5, 3], "random", heads=2)
    out, lse = oracle.Oracle(wl, sm_scale=0.0).attend()
    kv = f32(wl.kv_cache)
    k = 0
    for b in range(wl.bs):
        P, T = int(wl.prefix_lens[b]), int(wl.draft_lens[b])
        rows = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]],
                               wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]])
        blk = wl.mask_block(b).astype(bool)
        for i in range(T):
            vis_rows = rows[blk[i]]
            for h in range(wl.num_heads):
                np.testing.assert_allclose(out[k], kv[vis_rows, :W.D_V].mean(0), rtol=1e-13,
                                           atol=1e-14)
                assert abs(lse[k] - math.log(len(vis_rows))) < 1e-13
                k += 1


def test_no_visible_key():
    wl = small(91, [0], [3], "chain", heads=1)
    wl.custom_mask[:] = 0
    out, lse = oracle.Oracle(wl).attend()
    assert np.all(lse == -np.inf) and not out.any()


def test_bad_slot_is_reported():
    wl = small(92, [4], [2], "chain", heads=1)
    wl.kv_indices[1] = wl.num_slots + 3
    with pytest.raises(RuntimeError):
        oracle.Oracle(wl).attend()


def test_enumerate_matches_layout():
    wl = small(93, [6, 3], [3, 2], "random", heads=1)
    slots, vis = oracle.Oracle(wl).enumerate()
    off = 0
    for b in range(wl.bs):
        P, T = int(wl.prefix_lens[b]), int(wl.draft_lens[b])
        exp = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]],
                              wl.out_cache_loc[wl.qo_indptr[b]:wl.qo_indptr[b + 1]]])
        np.testing.assert_array_equal(slots[off:off + P + T], exp)
        blk = wl.mask_block(b)
        ev = blk.copy()
        ev[:, :P] = 1
        np.testing.assert_array_equal(vis[wl.mask_indptr[b]:wl.mask_indptr[b + 1]], ev.reshape(-1))
        off += P + T


# ---------------------------------------------------------------------------
# 7. The workspace figure of "The Architecture of Capture Safety" (section "Assumptions
#    and Their Validity", assumption 3): fp32 partial outputs of 512 dims, one per
#    (query token, head, split): bs 8 x 9 drafts x 64 heads x 64 splits.
# ---------------------------------------------------------------------------
def test_pages_workspace_figure():
    b = 8 * 9 * 64 * 64 * 512 * 4
    assert b == 603_979_776          # "about 600 MB" for batch size 8
    assert abs(b / 1e6 - 600) / 600 < 0.01


# ---------------------------------------------------------------------------
# 8. Hand-derived closed-form cases (tests/golden/closed_form_cases.json).
# ---------------------------------------------------------------------------
def _golden_workload(case):
    H = case["heads"]
    P = case["prefix_slots"]
    D = case["draft_slots"]
    pool = case["num_slots"]
    q = np.zeros((len(D), H, W.D_QK), dtype=np.float32)
    for (t, h, d, v) in case["q_nonzeros"]:
        q[t, h, d] = v
    kv = np.zeros((pool, W.D_QK), dtype=np.float32)
    for (s, d, v) in case["kv_nonzeros"]:
        kv[s, d] = v
    mask = np.array(case["mask"], dtype=np.uint8).reshape(-1)
    assert len(P) + len(D) == len(case["mask"][0])
    return W.Workload(
        name=case["name"], q=W._bf16_bits(q), kv_cache=W._bf16_bits(kv),
        kv_indices=np.array(P, dtype=np.int32), kv_indptr=np.array([0, len(P)], dtype=np.int32),
        out_cache_loc=np.array(D, dtype=np.int64), custom_mask=mask,
        mask_indptr=np.array([0, mask.shape[0]], dtype=np.int64),
        qo_indptr=np.array([0, len(D)], dtype=np.int64), parents=[], sm_scale=case["sm_scale"])


def _golden_cases():
    with open(os.path.join(GOLDEN, "closed_form_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_closed_form(case):
    wl = _golden_workload(case)
    out, lse = oracle.Oracle(wl).attend()
    out = out.reshape(wl.total_q, wl.num_heads, W.D_V)
    lse = lse.reshape(wl.total_q, wl.num_heads)
    ns = {"math": math, "__builtins__": {}}
    for e in case["expect"]:
        t, h = e["token"], e["head"]
        want = eval(e["lse"], ns)
        assert abs(lse[t, h] - want) < 1e-12, (e, lse[t, h])
        for d, expr in e["out_nonzeros"]:
            v = eval(expr, ns)
            assert abs(out[t, h, d] - v) < 1e-12, (d, out[t, h, d], v)
        nz = {d for d, _ in e["out_nonzeros"]}
        rest = [d for d in range(W.D_V) if d not in nz]
        assert np.all(out[t, h, rest] == 0.0)
