"""GPU parity of the 8-heads-per-token path (a tensor-parallel shard of 8 ranks).

With num_heads = 8 the kernel fills its 64 columns with the 8 heads of 8 consecutive
draft tokens of a request; the last group of a request may be short, and its columns past
the request's drafts must not be written.  Everything is compared with the fp64 oracle
(which is generic in the head count) at the same tolerance as the 64-head tests.
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
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))
    assert mtv.read_device_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("seed,P,T,tree", [
    (201, [0], [1], "chain"),                          # one token in a group of 8
    (202, [1, 127, 128, 129], [1, 8, 16, 3], "random"),  # full and short groups
    (203, [700, 0, 129, 50], [16, 3, 7, 9], "random"),   # ragged groups, several tiles
    (204, [2048, 300], [12, 16], "chain"),
])
def test_small_full(seed, P, T, tree):
    wl = W.build("tp8", seed, P, T, tree, 2 * (sum(P) + sum(T)) + 64, heads=8)
    _full_check(wl)


def test_rows_outside_the_batch_untouched():
    # q/out rows past qo_indptr[bs] (a short last group reads them as q, must not write)
    wl = W.build("tp8", 205, [90, 40], [3, 5], "random", 400, heads=8)
    d = to_device(wl)
    extra = 9
    q = torch.cat([d["q"], torch.randn((extra, 8, 576), device="cuda").to(torch.bfloat16)])
    d["q"] = q
    out, lse, ws, mq = alloc_outputs(wl)
    out = torch.full((wl.total_q + extra, 8, 512), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((wl.total_q + extra, 8), 7.0, dtype=torch.float32, device="cuda")
    mtv.mla_tree_verify(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                        d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], d["qo_indptr"],
                        wl.sm_scale, out, lse, ws, mq)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))
    assert (out[wl.total_q:].float() == 3.0).all() and (lse[wl.total_q:] == 7.0).all()


@pytest.mark.parametrize("shape_id", [2, 3, 4])
def test_shapes_sampled(shape_id):
    wl = W.shape(shape_id, heads=8)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    rows = sample_rows(wl, 64, seed=shape_id)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_index_dump_bit_exact():
    wl = W.build("tp8", 206, [300, 0, 129], [16, 3, 7], "random", 1024, heads=8)
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
    wl = W.shape(2, heads=8)
    d = to_device(wl)
    o1, l1, _ = run(wl, d)
    for _ in range(3):
        o2, l2, _ = run(wl, d)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_heads_8_and_64_agree_on_shared_heads():
    """Heads are independent: 8 of the 64 heads computed by the 64-head path agree with the
    8-head path on the same 8 heads, within the parity tolerance.  (Not bit for bit: the
    token grouping moves the CTA boundaries, so the partials are merged differently.)"""
    wl64 = W.build("h", 207, [500, 60], [16, 5], "random", 2048)
    wl8 = W.build("h", 207, [500, 60], [16, 5], "random", 2048)
    wl8.q = np.ascontiguousarray(wl64.q[:, 8:16, :])
    out64, lse64, _ = run(wl64)
    out8, lse8, _ = run(wl8)
    a = out64[:, 8:16].float().cpu().numpy().astype(np.float64)
    b = out8.float().cpu().numpy().astype(np.float64)
    assert (np.abs(a - b) / (1.0 + np.abs(a))).max() <= 1e-2
    assert np.abs(lse64[:, 8:16].cpu().numpy() - lse8.cpu().numpy()).max() <= 1e-3
