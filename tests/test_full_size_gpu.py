"""The verify configs at full size, in the launch configuration the benchmark times.

- configs 2 and 3: every (row, head) pair against the oracle;
- configs 4 and 5: every head of every query token whose keys are cut into more than
  one partial (so both merge paths are compared with the oracle at full size), plus a
  uniform sample of the others; the split tokens come from the work plan restated in
  Python (tests/test_plan_cpu.py), with the lanes the device planner recorded;
- config 4 once more with each merge path forced: the bits equal the normal call's.

Bar: |out - ref| <= 1e-2 (1 + |ref|) on the bf16 output and |lse - ref| <= 1e-3.
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
from test_plan_cpu import walk as walk_restated  # noqa: E402


def split_rows(wl, ws):
    """(row, head) pairs of every query token cut into more than one partial."""
    h = mtv.plan_header(ws)
    T = [int(x) for x in wl.draft_lens]
    L = [int(p) + int(t) for p, t in zip(wl.prefix_lens, wl.draft_lens)]
    gt = 64 // wl.num_heads
    segs, (_, _, U, C, groups, _) = walk_restated(T, L, mtv.split_grid(), h["lanes"], gt)
    assert (U, C) == (h["total_units"], h["capacity"])
    rows = set()
    for g, lane, b, cg, t0, t1, u0, slot, slots in segs:
        if len(slots) > 1:
            for t in range(cg * gt, min(T[b], (cg + 1) * gt)):
                rows.add(int(wl.qo_indptr[b]) + t)
    rows = sorted(rows)
    heads = np.arange(wl.num_heads)
    return np.array([[r, hh] for r in rows for hh in heads], dtype=np.int64).reshape(-1, 2)


@pytest.mark.parametrize("shape_id", [2, 3])
def test_every_row(shape_id):
    wl = W.shape(shape_id)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))


@pytest.mark.parametrize("shape_id", [4, 5])
def test_every_split_token_and_a_sample(shape_id):
    wl = W.shape(shape_id)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    rows = split_rows(wl, ws)
    assert len(rows) > 0
    h = mtv.plan_header(ws)
    assert h["merges_tmem"] + h["merges_ws"] == len(rows) // wl.num_heads
    rows = np.concatenate([rows, sample_rows(wl, 64, seed=shape_id)])
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(out, lse, ref_out, ref_lse, rows)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_forced_merge_paths_at_full_size():
    """Config 4 with every split token merged from the workspace (mode 1), and with the
    last piece's CTA merging from TMEM wherever it can (mode 2): the same bits as the
    normal call, which the test above checks against the oracle."""
    wl = W.shape(4)
    d = to_device(wl)
    res = {}
    for mode in (mtv.MERGE_AUTO, mtv.MERGE_NO_TMEM, mtv.MERGE_PREFER_TMEM):
        out, lse, ws, mq = alloc_outputs(wl)
        mtv.mla_tree_verify_debug_ex(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                                     d["out_cache_loc"], d["custom_mask"], d["mask_indptr"],
                                     d["qo_indptr"], wl.sm_scale, out, lse, ws, mq,
                                     merge_mode=mode)
        torch.cuda.synchronize()
        assert mtv.read_device_status(ws) == 0
        res[mode] = (out, lse, mtv.plan_header(ws))
    assert res[mtv.MERGE_NO_TMEM][2]["merges_tmem"] == 0
    assert res[mtv.MERGE_PREFER_TMEM][2]["merges_tmem"] > 0
    base_out, base_lse, _ = res[mtv.MERGE_AUTO]
    for mode in (mtv.MERGE_NO_TMEM, mtv.MERGE_PREFER_TMEM):
        out, lse, _ = res[mode]
        assert torch.equal(base_out.view(torch.int16), out.view(torch.int16))
        assert torch.equal(base_lse.view(torch.int32), lse.view(torch.int32))
