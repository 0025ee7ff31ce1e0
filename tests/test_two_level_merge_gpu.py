"""GPU parity of the two-level merge of long, split-heavy column groups.

A column group (one draft token at 64 heads, eight at 8 heads) cut into more than 16
pieces is merged in two levels: the last piece of each group of 8 merges the group into
one partial, and the last group merges those into the output (the split-K reduce of "The
Architecture of Capture Safety", section "The Design Emerges", done as two reduces).
These workloads are chosen so that the work plan, restated in Python
(tests/test_plan_cpu.py), cuts some column groups into 30 to 60 pieces, several of them
with a short last group, next to column groups merged in one level; every (row, head) pair
is compared with the fp64 oracle, and repeated calls must give the same bits.

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
from gpu_util import all_rows, check_rows, run, to_device  # noqa: E402
from test_plan_cpu import walk as walk_restated  # noqa: E402


def pieces_per_column_group(wl, ws):
    """{(request, column group): number of pieces} of the plan the device used."""
    h = mtv.plan_header(ws)
    T = [int(x) for x in wl.draft_lens]
    L = [int(p) + int(t) for p, t in zip(wl.prefix_lens, wl.draft_lens)]
    segs, (_, _, U, C, _, _) = walk_restated(T, L, mtv.split_grid(), h["lanes"],
                                              64 // wl.num_heads)
    assert (U, C) == (h["total_units"], h["capacity"])
    return {(b, cg): len(slots) for _, _, b, cg, _, _, _, _, slots in segs}


@pytest.mark.parametrize("name,P,T,heads,short_group", [
    ("one token, 51 pieces", [26000], [1], 64, True),
    ("30 and 60 pieces", [60000, 30000], [1, 2], 64, True),
    ("53 pieces beside a one-level group", [40000, 9000], [1, 1], 64, True),
    ("17 pieces: a last group of one", [8250], [1], 64, True),
    ("24 pieces: three full groups", [12000], [1], 64, False),
    ("25 pieces", [12500], [1], 64, True),
])
def test_every_row(name, P, T, heads, short_group):
    wl = W.build("two-level", 301 + len(P), P, T, "chain", 2 * (sum(P) + sum(T)) + 64,
                 heads=heads)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    n = pieces_per_column_group(wl, ws)
    assert max(n.values()) > 16, n
    assert any(v > 16 and v % 8 for v in n.values()) == short_group, n
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))
    h = mtv.plan_header(ws)
    assert h["merges_tmem"] + h["merges_ws"] == sum(1 for v in n.values() if v > 1)


def test_long_context_at_8_heads_every_row():
    """The long-context config at 8 heads: both column groups in 58 pieces."""
    wl = W.shape(3, heads=8)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    n = pieces_per_column_group(wl, ws)
    assert min(n.values()) > 16, n
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))


def test_deterministic_repeat():
    wl = W.build("two-level", 310, [60000, 30000], [1, 2], "chain", 180128)
    d = to_device(wl)
    o1, l1, ws = run(wl, d)
    assert max(pieces_per_column_group(wl, ws).values()) > 16
    for _ in range(3):
        o2, l2, _ = run(wl, d)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
