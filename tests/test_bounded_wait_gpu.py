"""Failure detection inside the split kernel, without a GPU fault.

Every pipeline wait in the split kernel is bounded.  Here one small call runs with the
bound lowered to 1 microsecond (mla_tree_verify_debug_ex's wait_limit_ns), which the
first waits for q and key rows from memory cannot meet: the kernel must report
MLA_TV_DEV_TIMEOUT, drain its copies and MMAs, free its tensor memory and return, and
the next normal call on the same workspace must be correct.
"""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import workloads as W  # noqa: E402
from gpu_util import all_rows, alloc_outputs, check_rows, to_device  # noqa: E402


def test_expired_wait_reports_and_the_next_call_is_correct():
    wl = W.build("wait", 501, [3000, 700], [16, 8], "random", 8192)
    d = to_device(wl)
    out, lse, ws, mq = alloc_outputs(wl)
    args = (d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"],
            d["custom_mask"], d["mask_indptr"], d["qo_indptr"], wl.sm_scale, out, lse, ws, mq)
    mtv.mla_tree_verify_debug_ex(*args, wait_limit_ns=1000)
    torch.cuda.synchronize()
    assert mtv.read_device_status(ws) & mtv.DEV_TIMEOUT
    # the context and the workspace are still usable
    out.fill_(float("nan"))
    mtv.mla_tree_verify(*args)
    torch.cuda.synchronize()
    assert mtv.read_device_status(ws) == 0
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))
