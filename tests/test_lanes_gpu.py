"""The lane-group work plan on the GPU: every lane choice against the oracle, the device
planner against the plan restated in Python, and the two merge paths.

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
from gpu_util import all_rows, alloc_outputs, check_rows, to_device  # noqa: E402
from test_plan_cpu import plan as plan_restated  # noqa: E402


def call(wl, d, lanes=0, merge_mode=mtv.MERGE_AUTO, max_q=None):
    out, lse, ws, mq = alloc_outputs(wl, max_q)
    mtv.mla_tree_verify_debug_ex(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                                 d["out_cache_loc"], d["custom_mask"], d["mask_indptr"],
                                 d["qo_indptr"], wl.sm_scale, out, lse, ws, mq,
                                 merge_mode=merge_mode, lanes=lanes)
    torch.cuda.synchronize()
    return out, lse, ws


WORKLOADS = [
    ("ragged", 401, [0, 37, 300, 1000, 129], [4, 5, 16, 1, 3], "random", 64),
    ("chain", 402, [2048, 5, 700], [9, 16, 2], "chain", 64),
    ("long", 403, [20000, 60], [16, 7], "random", 64),
    ("heads8", 404, [900, 40, 3000], [37, 9, 16], "random", 8),
]


@pytest.mark.parametrize("lanes", [1, 2, 4, 8])
@pytest.mark.parametrize("case", WORKLOADS, ids=[w[0] for w in WORKLOADS])
def test_every_lane_choice_matches_the_oracle(case, lanes):
    name, seed, P, T, tree, heads = case
    wl = W.build(name, seed, P, T, tree, 2 * (sum(P) + sum(T)) + 64, heads=heads)
    d = to_device(wl)
    out, lse, ws = call(wl, d, lanes=lanes)
    assert mtv.read_device_status(ws) == 0
    h = mtv.plan_header(ws)
    assert h["lanes"] == lanes and h["groups"] == mtv.split_grid() // lanes
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))


@pytest.mark.parametrize("shape_id", [1, 2, 3, 4])
def test_device_plan_matches_the_restated_plan(shape_id):
    """The planner's units and capacity equal those of the plan restated in Python (with
    the lanes the library chose), and each lane choice keeps the capacity rule."""
    wl = W.shape(shape_id)
    d = to_device(wl)
    T = [int(x) for x in wl.draft_lens]
    L = [int(p) + int(t) for p, t in zip(wl.prefix_lens, wl.draft_lens)]
    grid = mtv.split_grid()
    for lanes in (0, 1, 8):
        out, lse, ws = call(wl, d, lanes=lanes)
        h = mtv.plan_header(ws)
        _, cum, U, C, groups, _ = plan_restated(T, L, grid, h["lanes"])
        assert (h["total_units"], h["capacity"], h["groups"]) == (U, C, groups)


@pytest.mark.parametrize("shape_id", [2, 4])
def test_merge_paths_give_the_same_bits(shape_id):
    """Merge mode 1 merges every split token from the workspace, mode 2 merges from TMEM
    wherever the last piece's CTA can wait for the others; the output bits do not depend
    on the path, and both paths ran (the header counts them)."""
    wl = W.shape(shape_id)
    d = to_device(wl)
    o0, l0, ws0 = call(wl, d)
    o1, l1, ws1 = call(wl, d, merge_mode=mtv.MERGE_NO_TMEM)
    o2, l2, ws2 = call(wl, d, merge_mode=mtv.MERGE_PREFER_TMEM)
    h1, h2 = mtv.plan_header(ws1), mtv.plan_header(ws2)
    assert h1["merges_tmem"] == 0 and h1["merges_ws"] > 0
    assert h2["merges_tmem"] > 0
    for o, l in ((o1, l1), (o2, l2)):
        assert torch.equal(o0.view(torch.int16), o.view(torch.int16))
        assert torch.equal(l0.view(torch.int32), l.view(torch.int32))
