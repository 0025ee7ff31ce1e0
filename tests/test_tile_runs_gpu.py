"""GPU parity of the tile loads for runs of consecutive slots.

When the request's prefix may be one run of consecutive slots (its first and last slots
P - 1 apart) and all 128 rows of a key tile sit in consecutive pool slots (a defragmented
prefix), the split kernel loads each chunk of the tile with one TMA tile copy instead of
128 row copies; any other tile is gathered row by row.  The two loads must fill shared memory
identically, so a workload whose rows are laid out consecutively (or in runs) must give
bit for bit the output of the same workload with scattered rows, and both must match the
oracle.
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
from gpu_util import all_rows, check_rows, run, sample_rows  # noqa: E402


def _same_bits(a, b):
    oa, la, wa = a
    ob, lb, wb = b
    assert mtv.read_device_status(wa) == 0 and mtv.read_device_status(wb) == 0
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)


@pytest.mark.parametrize("seed,P,T,tree", [
    (301, [128], [1], "chain"),                       # one full tile, nothing else
    (302, [127, 128, 129, 255, 256, 257], [1, 3, 16, 16, 2, 9], "random"),   # ragged tails
    (303, [1000, 4000, 0, 300], [16, 16, 5, 16], "random"),
    (304, [5000], [16], "chain"),
])
@pytest.mark.parametrize("layout", ["contiguous", "runs"])
def test_small_full_and_bit_identical(seed, P, T, tree, layout):
    pool = 4 * (sum(P) + sum(T)) + 4096
    wl_s = W.build("s", seed, P, T, tree, pool)
    wl_c = W.build("c", seed, P, T, tree, pool, layout=layout)
    got = run(wl_c)
    ref_out, ref_lse = oracle.Oracle(wl_c).attend()
    check_rows(got[0], got[1], ref_out, ref_lse, all_rows(wl_c))
    _same_bits(got, run(wl_s))


@pytest.mark.parametrize("shape_id", [2, 3, 4])
def test_shapes_contiguous(shape_id):
    wl = W.shape(shape_id, layout="contiguous")
    got = run(wl)
    rows = sample_rows(wl, 64, seed=shape_id)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows)
    check_rows(got[0], got[1], ref_out, ref_lse, rows)
    _same_bits(got, run(W.shape(shape_id)))


def test_slot_zero_and_pool_end():
    # a run that starts at slot 0 and one that ends at the last slot of the pool
    wl = W.build("edge", 305, [256, 384], [4, 4], "chain", 648, layout="contiguous", poison=True)
    n = 256 + 4 + 384 + 4
    assert n == 648
    got = run(wl)
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(got[0], got[1], ref_out, ref_lse, all_rows(wl))
    _same_bits(got, run(W.build("edge", 305, [256, 384], [4, 4], "chain", 648)))


def test_heads_8_contiguous():
    wl = W.build("tp8", 306, [700, 129, 2048], [16, 7, 9], "random", 12000, heads=8,
                 layout="contiguous")
    got = run(wl)
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(got[0], got[1], ref_out, ref_lse, all_rows(wl))
    _same_bits(got, run(W.build("tp8", 306, [700, 129, 2048], [16, 7, 9], "random", 12000,
                                heads=8)))
