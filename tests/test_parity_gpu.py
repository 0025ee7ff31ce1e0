"""Parity of the CUDA path with the fp64 oracle, called through the C ABI.

Bar: |out - ref| <= 1e-2 (1 + |ref|) on the bf16 output and |lse - ref| <= 1e-3;
gathered slots and mask bits bit-exact against the oracle's enumeration.  Every
workload's pool holds bf16 NaN in each slot no request references, so a stray gather
shows up as a non-finite output.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import workloads as W  # noqa: E402
from gpu_util import all_rows, alloc_outputs, check_rows, run, sample_rows, to_device  # noqa: E402


def _full_check(wl, **kw):
    out, lse, ws = run(wl, **kw)
    ref_out, ref_lse = oracle.Oracle(wl, sm_scale=kw.get("sm_scale")).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))
    assert mtv.read_device_status(ws) == 0
    return out, lse


def test_shape1_full():
    _full_check(W.shape(1))


@pytest.mark.parametrize("seed,P,T,tree", [
    (101, [0], [1], "chain"),                     # one key: the token itself
    (102, [1, 127, 128, 129], [1, 1, 16, 3], "random"),   # around one tile
    (103, [0, 37, 300, 1000], [4, 5, 16, 1], "random"),   # several tiles, ragged tails
    (104, [511, 2], [16, 16], "chain"),
    (105, [2048], [8], "random"),
])
def test_small_full(seed, P, T, tree):
    wl = W.build("t", seed, P, T, tree, 2 * (sum(P) + sum(T)) + 64)
    _full_check(wl)


def test_max_q_larger_than_needed():
    wl = W.build("t", 106, [70, 5], [3, 2], "random", 200)
    _full_check(wl, max_q_per_req=16)


def test_zero_draft_request_and_offset_rows():
    """A request with T_b = 0 in the middle; rows of q/out past qo_indptr[bs] untouched."""
    wl = W.build("t", 107, [40, 33, 90], [3, 1, 4], "random", 400)
    # drop request 1's single draft: T_1 = 0, its mask block empty
    P = wl.prefix_lens
    q0, q1 = int(wl.qo_indptr[1]), int(wl.qo_indptr[2])
    keep = np.r_[0:q0, q1:wl.total_q]
    wl.q = wl.q[keep]
    wl.out_cache_loc = wl.out_cache_loc[keep]
    m0, m1 = int(wl.mask_indptr[1]), int(wl.mask_indptr[2])
    wl.custom_mask = np.concatenate([wl.custom_mask[:m0], wl.custom_mask[m1:]])
    wl.qo_indptr = np.array([0, 3, 3, 7], dtype=np.int64)
    wl.mask_indptr = np.array([0, m0, m0, m0 + (wl.custom_mask.shape[0] - m0)], dtype=np.int64)
    _full_check(wl)


def test_mask_only_diagonal_and_no_prefix():
    wl = W.build("t", 108, [0, 0], [16, 7], "random", 100)
    for b in range(wl.bs):
        blk = wl.mask_block(b)
        blk[...] = 0
        np.fill_diagonal(blk, 1)
    out, lse = _full_check(wl)
    # one visible key: the output is that key's V row rounded to bf16
    kv = torch.from_numpy(wl.kv_cache.view(np.int16)).view(torch.bfloat16)
    for r in range(wl.total_q):
        exp = kv[int(wl.out_cache_loc[r]), :512].float()
        assert torch.equal(out[r].float().cpu(), exp.expand(wl.num_heads, -1))


def test_all_masked_row_gives_minus_inf():
    wl = W.build("t", 109, [0], [4], "chain", 50)
    blk = wl.mask_block(0)
    blk[2, :] = 0       # draft 2 sees nothing
    _full_check(wl)


def test_outliers_and_scaled_inputs():
    wl = W.build("t", 110, [3000, 700], [8, 16], "random", 8192, q_scale=0.5, kv_scale=0.5,
                 outlier_frac=0.01, outlier_mult=8.0)
    _full_check(wl)


def test_index_dump_bit_exact():
    wl = W.build("t", 111, [300, 0, 129], [16, 3, 7], "random", 1024)
    d = to_device(wl)
    out, lse, ws, mq = alloc_outputs(wl)
    L = int((wl.prefix_lens + wl.draft_lens).sum())
    slot_dump = torch.full((L,), -7, dtype=torch.int64, device="cuda")
    vis_dump = torch.full((wl.custom_mask.shape[0],), 9, dtype=torch.uint8, device="cuda")
    mtv.mla_tree_verify_debug(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                              d["out_cache_loc"], d["custom_mask"], d["mask_indptr"],
                              d["qo_indptr"], wl.sm_scale, out, lse, ws, mq, slot_dump, vis_dump)
    torch.cuda.synchronize()
    slots, vis = oracle.Oracle(wl).enumerate()
    np.testing.assert_array_equal(slot_dump.cpu().numpy(), slots)
    np.testing.assert_array_equal(vis_dump.cpu().numpy(), vis)


def test_deterministic_repeat():
    # Which CTA merges a split token, and whether it merges from TMEM or from the
    # workspace, depends on timing; the bits must not.
    wl = W.build("t", 112, [900, 50], [16, 4], "random", 4096)
    d = to_device(wl)
    o1, l1, _ = run(wl, d)
    for _ in range(4):
        o2, l2, _ = run(wl, d)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    wl = W.shape(2)
    d = to_device(wl)
    o1, l1, _ = run(wl, d)
    for _ in range(3):
        o2, l2, _ = run(wl, d)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("shape_id", [2, 3, 4, 5])
def test_shapes_sampled(shape_id):
    """The five verify shapes at full size, in the launch configuration the benchmark
    times; the oracle computes a sample of (row, head) pairs one by one."""
    wl = W.shape(shape_id)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    rows = sample_rows(wl, 48, seed=shape_id)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)
    # properties at any size: every row of the batch written, finite
    assert torch.isfinite(out.float()).all()
    assert torch.isfinite(lse).all()


def test_bad_slot_sets_flag_without_fault():
    wl = W.build("t", 113, [50], [4], "chain", 200)
    wl.kv_indices[10] = wl.num_slots + 5     # outside the pool
    wl.out_cache_loc[1] = -3
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) & mtv.DEV_BAD_SLOT


def test_bad_indptr_sets_flag():
    wl = W.build("t", 114, [50, 20], [4, 2], "chain", 200)
    wl.kv_indptr[1] = 1000                    # beyond kv_indices
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) & mtv.DEV_BAD_INDPTR


def test_bad_mask_indptr_zeroes_request():
    wl = W.build("t", 115, [50, 20], [4, 2], "chain", 200)
    wl.mask_indptr[2] += 1                    # request 1's block has the wrong length
    wl.custom_mask = np.concatenate([wl.custom_mask, np.ones(1, np.uint8)])
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) & mtv.DEV_BAD_MASK
    assert torch.all(lse[4:6] == -np.inf) and not out[4:6].float().abs().sum()
    ref_out, ref_lse = oracle.Oracle(wl).attend(all_rows(wl)[: 4 * wl.num_heads])
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl)[: 4 * wl.num_heads])


def test_graph_capture_replay_with_new_contents():
    """Capture one call on static buffers, then rewrite their contents (same addresses,
    same sizes) and replay: each replay computes the batch now in the buffers."""
    wl_a = W.build("a", 116, [1500, 300], [16, 8], "random", 8192)
    wl_b = W.build("b", 117, [1500, 300], [16, 8], "random", 8192)
    src = {"a": to_device(wl_a), "b": to_device(wl_b)}
    st = {k: v.clone() for k, v in src["a"].items()}
    out, lse, ws, mq = alloc_outputs(wl_a)
    mtv.prepare()
    s = torch.cuda.Stream()

    def call():
        mtv.mla_tree_verify(st["q"], st["kv_cache"], st["kv_indices"], st["kv_indptr"],
                            st["out_cache_loc"], st["custom_mask"], st["mask_indptr"],
                            st["qo_indptr"], wl_a.sm_scale, out, lse, ws, mq, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for name, wl in (("b", wl_b), ("a", wl_a), ("b", wl_b)):
        for k in st:
            st[k].copy_(src[name][k])
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        rows = sample_rows(wl, 64, seed=3)
        ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
        check_rows(out, lse, ref_out, ref_lse, rows)
    assert mtv.read_device_status(ws) == 0


def test_shape5_graph_replay_with_new_q():
    """The mixed-T outlier shape at full size (64 requests, 8k-64k prefixes, a 4M-slot
    pool) runs as a CUDA-graph replay of one captured call; the second replay sees new
    q contents in the same buffer (every token's q moved one row down)."""
    import dataclasses
    wl = W.shape(5)
    d = to_device(wl)
    out, lse, ws, mq = alloc_outputs(wl)
    mtv.prepare()
    s = torch.cuda.Stream()

    def call():
        mtv.mla_tree_verify(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                            d["out_cache_loc"], d["custom_mask"], d["mask_indptr"],
                            d["qo_indptr"], wl.sm_scale, out, lse, ws, mq, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for variant in (0, 1):
        wlv = wl
        if variant == 1:
            q2 = np.ascontiguousarray(np.roll(wl.q, 1, axis=0))
            d["q"].copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16))
            wlv = dataclasses.replace(wl, q=q2)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert mtv.read_device_status(ws) == 0
        rows = sample_rows(wlv, 32, seed=50 + variant)
        ref_out, ref_lse = oracle.Oracle(wlv).attend(rows)
        check_rows(out, lse, ref_out, ref_lse, rows)
        assert torch.isfinite(out.float()).all()


def test_many_requests_planner_passes():
    """1500 requests (more than one pass of the 1024-thread planner's scan), with short
    and empty prefixes and 0-3 drafts each; sampled rows against the oracle and every
    row written."""
    rng = np.random.default_rng(120)
    bs = 1500
    P = rng.integers(0, 300, size=bs)
    T = rng.integers(0, 4, size=bs)
    T[0] = 1
    wl = W.build("many", 120, P, T, "random", int(P.sum() + T.sum()) + 512)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    rows = sample_rows(wl, 96, seed=120)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_more_than_32_bad_mask_blocks():
    """40 of 60 requests have a mask block of the wrong length: their rows become
    0 / -inf (the planner's path for more than 32 such requests) and the other rows
    stay correct."""
    bs = 60
    wl = W.build("badm", 121, [40] * bs, [2] * bs, "chain", 8192)
    L = 42
    bad = list(range(0, 40))
    # rebuild mask_indptr so that bad requests' blocks are one byte too long
    lengths = np.array([2 * L + (1 if b in bad else 0) for b in range(bs)], dtype=np.int64)
    new_ptr = np.zeros(bs + 1, dtype=np.int64)
    new_ptr[1:] = np.cumsum(lengths)
    new_mask = np.ones(int(new_ptr[-1]), dtype=np.uint8)
    for b in range(bs):
        blk = wl.custom_mask[wl.mask_indptr[b]:wl.mask_indptr[b + 1]]
        new_mask[new_ptr[b]:new_ptr[b] + blk.size] = blk
    wl.mask_indptr = new_ptr
    wl.custom_mask = new_mask
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) & mtv.DEV_BAD_MASK
    for b in range(bs):
        r0, r1 = int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1])
        if b in bad:
            assert torch.all(lse[r0:r1] == -np.inf) and not out[r0:r1].float().abs().sum()
    good = [b for b in range(bs) if b not in bad]
    rows = np.array([[r, h] for b in good[:5] for r in range(int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1]))
                     for h in (0, 31, 63)])
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)


@pytest.mark.parametrize("seed,P,T,tree", [
    (130, [300, 1000], [33, 64], "random"),      # trees larger than the configs' 16 tokens
    (131, [0, 129], [40, 17], "chain"),
])
def test_larger_trees_full(seed, P, T, tree):
    """Up to 64 draft tokens per request (the C ABI takes up to 4096): every row against
    the oracle."""
    wl = W.build("big_t", seed, P, T, tree, 2 * (sum(P) + sum(T)) + 64)
    _full_check(wl)


def test_long_chain_sampled():
    """A 200-token draft chain over a 500-key prefix: the draft block alone spans two key
    tiles; sampled rows against the oracle, every row finite."""
    wl = W.build("chain200", 132, [500], [200], "chain", 1500)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    rows = sample_rows(wl, 128, seed=132)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_larger_tree_heads_8():
    """8 heads per token with 37 draft tokens: 5 token groups, the last one short."""
    wl = W.build("big_t8", 133, [260, 40], [37, 9], "random", 800, heads=8)
    _full_check(wl)
