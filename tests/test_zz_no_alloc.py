"""The entry point that allocates nothing, checked against the one that takes a workspace.

mla_tree_verify_static_ws() serves callers that cannot allocate device memory (for
example an engine that keeps its memory pool private, or C code that may not call
cudaMalloc on this path because it can synchronise the device and is not allowed during
graph capture).  It uses a scratch array built into the library instead of a
caller-provided workspace.  Here it is called through the C ABI twice in a row, on
different batches (64 and 8 heads), and each result must equal the workspace entry
point's result for the same batch bit for bit: both run the same kernels on the same
work plan.  It is also captured in a CUDA graph after mla_tree_verify_prepare() and
replayed.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import binding  # noqa: E402
from mla_tree_verify_gb300 import workloads as W  # noqa: E402
from gpu_util import alloc_outputs, to_device  # noqa: E402

STATIC_LIMIT = -9


def _lib():
    lib = binding.load()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.mla_tree_verify_static_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                              vp, vp, i32, i32, i32, i64, i64, i64, i64, vp]
    lib.mla_tree_verify_static_ws.restype = ctypes.c_int
    return lib


def _call_static(lib, wl, d, out, lse, mq, stream=None):
    stream = ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
    return lib.mla_tree_verify_static_ws(
        d["q"].data_ptr(), d["kv_cache"].data_ptr(), d["kv_indices"].data_ptr(),
        d["kv_indptr"].data_ptr(), d["out_cache_loc"].data_ptr(), d["custom_mask"].data_ptr(),
        d["mask_indptr"].data_ptr(), d["qo_indptr"].data_ptr(), ctypes.c_float(wl.sm_scale),
        out.data_ptr(), lse.data_ptr(), wl.bs, mq, wl.num_heads, wl.num_slots, wl.total_q,
        d["kv_indices"].numel(), d["custom_mask"].numel(), stream)


def _with_workspace(wl, d):
    out, lse, ws, mq = alloc_outputs(wl)
    mtv.mla_tree_verify(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                        d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], d["qo_indptr"],
                        wl.sm_scale, out, lse, ws, mq)
    torch.cuda.synchronize()
    return out, lse


def _same(a_out, a_lse, b_out, b_lse):
    b = b_out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(b))
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse.view(torch.int32), b_lse.view(torch.int32))


def test_static_scratch_matches_workspace_entry_twice_in_a_row():
    lib = _lib()
    batches = [W.build("a", 301, [700, 0, 129], [16, 3, 7], "random", 2048),
               W.shape(2),
               W.build("h8", 303, [900, 40], [16, 5], "random", 2048, heads=8)]
    for wl in batches:   # two calls in a row, different sizes, shared scratch
        d = to_device(wl)
        ref_out, ref_lse = _with_workspace(wl, d)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _call_static(lib, wl, d, out, lse, wl.max_q_per_req)
        assert st == 0, lib.mla_tree_verify_status_string(st)
        torch.cuda.synchronize()
        _same(ref_out, ref_lse, out, lse)


def test_static_scratch_in_a_captured_graph():
    """prepare() looks up the scratch array's address, so the first static call may be
    the one captured; the replay must give the workspace entry point's bits."""
    lib = _lib()
    assert lib.mla_tree_verify_prepare() == 0
    wl = W.build("g", 304, [1500, 300], [16, 8], "random", 4096)
    d = to_device(wl)
    ref_out, ref_lse = _with_workspace(wl, d)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = _call_static(lib, wl, d, out, lse, wl.max_q_per_req, stream=s)
    assert st == 0, lib.mla_tree_verify_status_string(st)
    for _ in range(2):
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        _same(ref_out, ref_lse, out, lse)


def test_static_scratch_rejects_a_batch_beyond_its_size():
    lib = _lib()
    wl = W.build("c", 302, [40], [4], "chain", 100)
    d = to_device(wl)
    out = torch.zeros((wl.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((wl.total_q, 64), dtype=torch.float32, device="cuda")
    # 64 requests x 4096 drafts need far more than the built-in scratch holds
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.mla_tree_verify_static_ws(
        d["q"].data_ptr(), d["kv_cache"].data_ptr(), d["kv_indices"].data_ptr(),
        d["kv_indptr"].data_ptr(), d["out_cache_loc"].data_ptr(), d["custom_mask"].data_ptr(),
        d["mask_indptr"].data_ptr(), d["qo_indptr"].data_ptr(), ctypes.c_float(wl.sm_scale),
        out.data_ptr(), lse.data_ptr(), 64, 4096, 64, wl.num_slots, wl.total_q,
        d["kv_indices"].numel(), d["custom_mask"].numel(), stream)
    assert st == STATIC_LIMIT
    assert lib.mla_tree_verify_status_string(st).decode().startswith("batch needs more scratch")
