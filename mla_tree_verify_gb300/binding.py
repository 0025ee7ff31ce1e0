"""Thin Python binding of libmla_tree_verify.so (include/mla_tree_verify.h).

Argument marshalling only: torch tensors are checked for dtype, shape and device and
their data pointers, together with sizes and the raw CUDA stream handle, are passed
to the C entry points of the same names.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback, and importing this module on a machine
without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

HEADS = 64
D_QK = 576
D_V = 512
NSPLIT = 64

_STATUS = {
    0: "ok", -1: "null pointer", -2: "num_heads must be 64", -3: "bad shape",
    -4: "misaligned buffer", -5: "workspace too small", -6: "launch failed",
    -7: "no sm_103 device", -8: "sm_scale not finite",
}
DEV_BAD_SLOT = 1
DEV_BAD_INDPTR = 2
DEV_BAD_MASK = 4
DEV_TIMEOUT = 8

_lib = None


class MlaTreeVerifyError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Loads the shared library (built beforehand by build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with mla_tree_verify_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    common = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, i32, i32, i32,
              i64, i64, i64, i64]
    lib.mla_tree_verify.argtypes = common + [vp]
    lib.mla_tree_verify.restype = ctypes.c_int
    lib.mla_tree_verify_debug.argtypes = common + [vp, vp, vp]
    lib.mla_tree_verify_debug.restype = ctypes.c_int
    lib.mla_tree_verify_debug_ex.argtypes = common + [ctypes.POINTER(DebugOpts), vp]
    lib.mla_tree_verify_debug_ex.restype = ctypes.c_int
    lib.mla_tree_verify_profiled.argtypes = common + [vp, vp]
    lib.mla_tree_verify_profiled.restype = ctypes.c_int
    lib.mla_tree_verify_workspace_bytes.argtypes = [i32, i32, i32]
    lib.mla_tree_verify_workspace_bytes.restype = sz
    lib.mla_tree_verify_prepare.argtypes = []
    lib.mla_tree_verify_prepare.restype = ctypes.c_int
    lib.mla_tree_verify_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.mla_tree_verify_read_device_status.restype = ctypes.c_int
    lib.mla_tree_verify_split_grid.argtypes = []
    lib.mla_tree_verify_split_grid.restype = i32
    lib.mla_tree_verify_kv_gather.argtypes = [vp, i64, vp, i64, vp, i32, vp, i64, i32, vp, vp,
                                              vp]
    lib.mla_tree_verify_kv_gather.restype = ctypes.c_int
    lib.causal_conv1d_update_dedup.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                               i32, i64, i32, vp]
    lib.causal_conv1d_update_dedup.restype = ctypes.c_int
    lib.causal_conv1d_update_dedup_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                                  i32, i32, i64, i32, i32, i32, vp, vp, vp]
    lib.causal_conv1d_update_dedup_ex.restype = ctypes.c_int
    lib.mla_tree_verify_status_string.argtypes = [ctypes.c_int]
    lib.mla_tree_verify_status_string.restype = ctypes.c_char_p
    if path == _build.LIB:
        _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load().mla_tree_verify_status_string(status).decode()
        raise MlaTreeVerifyError(f"mla_tree_verify status {status}: {msg}")


def workspace_bytes(bs: int, max_q_per_req: int, num_heads: int = HEADS) -> int:
    n = load().mla_tree_verify_workspace_bytes(bs, max_q_per_req, num_heads)
    if n == 0:
        raise MlaTreeVerifyError("invalid workspace query")
    return int(n)


def prepare() -> None:
    _check(load().mla_tree_verify_prepare())


def split_grid() -> int:
    return int(load().mla_tree_verify_split_grid())


class DebugOpts(ctypes.Structure):
    """mla_tree_verify_debug_opts of include/mla_tree_verify.h."""
    _fields_ = [("slot_dump", ctypes.c_void_p), ("vis_dump", ctypes.c_void_p),
                ("wait_limit_ns", ctypes.c_uint64), ("merge_mode", ctypes.c_int32),
                ("lanes", ctypes.c_int32)]


MERGE_AUTO = 0
MERGE_NO_TMEM = 1
MERGE_PREFER_TMEM = 2


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _args(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr, qo_indptr,
          sm_scale, out, lse, workspace, max_q_per_req):
    import torch
    checks = [
        (q, torch.bfloat16, 3), (kv_cache, torch.bfloat16, 2), (kv_indices, torch.int32, 1),
        (kv_indptr, torch.int32, 1), (out_cache_loc, torch.int64, 1),
        (custom_mask, torch.uint8, 1), (mask_indptr, torch.int64, 1), (qo_indptr, torch.int64, 1),
        (out, torch.bfloat16, 3), (lse, torch.float32, 2), (workspace, torch.uint8, 1),
    ]
    for t, dt, nd in checks:
        if t.dtype != dt or t.dim() != nd or not t.is_contiguous() or not t.is_cuda:
            raise MlaTreeVerifyError(f"expected a contiguous CUDA {dt} tensor with {nd} dims, "
                                     f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    bs = kv_indptr.shape[0] - 1
    if q.shape[2] != D_QK:
        raise MlaTreeVerifyError(f"q must be [total_q, 64, 576], got {tuple(q.shape)}")
    if kv_cache.shape[1] != D_QK or out.shape[1:] != (q.shape[1], D_V):
        raise MlaTreeVerifyError("kv_cache must be [slots, 576] and out [total_q, H, 512]")
    if out.shape[0] != q.shape[0] or lse.shape != (q.shape[0], q.shape[1]):
        raise MlaTreeVerifyError("out/lse rows must match q")
    if max_q_per_req is None:
        raise MlaTreeVerifyError("max_q_per_req is required (it fixes the launch grid)")
    return [q.data_ptr(), kv_cache.data_ptr(), kv_indices.data_ptr(), kv_indptr.data_ptr(),
            out_cache_loc.data_ptr(), custom_mask.data_ptr(), mask_indptr.data_ptr(),
            qo_indptr.data_ptr(), ctypes.c_float(sm_scale), out.data_ptr(), lse.data_ptr(),
            workspace.data_ptr(), workspace.numel(), bs, int(max_q_per_req), q.shape[1],
            kv_cache.shape[0], q.shape[0], kv_indices.numel(), custom_mask.numel()]


def mla_tree_verify(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
                    qo_indptr, sm_scale, out, lse, workspace, max_q_per_req, stream=None):
    """Enqueues the verify attention on ``stream`` (default: torch's current stream).

    All tensors live on the device: q bf16 [total_q, 64, 576], kv_cache bf16
    [slots, 576], kv_indices int32, kv_indptr int32 [bs+1], out_cache_loc int64
    [total_q], custom_mask uint8, mask_indptr int64 [bs+1], qo_indptr int64 [bs+1],
    out bf16 [total_q, 64, 512], lse fp32 [total_q, 64], workspace uint8 of at least
    workspace_bytes(bs, max_q_per_req) bytes.  Nothing is synchronised."""
    a = _args(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
              qo_indptr, sm_scale, out, lse, workspace, max_q_per_req)
    _check(load().mla_tree_verify(*a, _stream_handle(stream)))


def mla_tree_verify_debug(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask,
                          mask_indptr, qo_indptr, sm_scale, out, lse, workspace, max_q_per_req,
                          slot_dump, vis_dump, stream=None):
    """As mla_tree_verify, also recording the gathered slot of every key column
    (slot_dump int64 [sum_b L_b]) and the visibility used for every mask entry
    (vis_dump uint8 [mask length])."""
    import torch
    a = _args(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
              qo_indptr, sm_scale, out, lse, workspace, max_q_per_req)
    if slot_dump.dtype != torch.int64 or vis_dump.dtype != torch.uint8:
        raise MlaTreeVerifyError("slot_dump must be int64 and vis_dump uint8")
    _check(load().mla_tree_verify_debug(*a, slot_dump.data_ptr(), vis_dump.data_ptr(),
                                        _stream_handle(stream)))


def mla_tree_verify_debug_ex(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask,
                             mask_indptr, qo_indptr, sm_scale, out, lse, workspace,
                             max_q_per_req, slot_dump=None, vis_dump=None, wait_limit_ns=0,
                             merge_mode=MERGE_AUTO, lanes=0, stream=None):
    """As mla_tree_verify, with the debug settings of mla_tree_verify_debug_ex(): optional
    index dumps (both or neither), the limit of the split kernel's bounded waits (0: the
    default 2 s), which path merges the partials (MERGE_*), and the CTAs per lane group
    (0: the library's choice)."""
    a = _args(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
              qo_indptr, sm_scale, out, lse, workspace, max_q_per_req)
    opts = DebugOpts(slot_dump.data_ptr() if slot_dump is not None else None,
                     vis_dump.data_ptr() if vis_dump is not None else None,
                     int(wait_limit_ns), int(merge_mode), int(lanes))
    _check(load().mla_tree_verify_debug_ex(*a, ctypes.byref(opts), _stream_handle(stream)))


def plan_header(workspace) -> dict:
    """The work plan's header as the planner wrote it into ``workspace`` (synchronises):
    total units, units per lane group (capacity), largest tile count, lanes and groups,
    and how many split query tokens (column groups) were merged from TMEM and how many
    from the workspace."""
    import numpy as np
    h = workspace[:56].cpu().numpy()
    i32, i64 = h.view(np.int32), h.view(np.int64)
    return {"error_flags": int(i32[0]), "grid": int(i32[1]), "total_units": int(i64[1]),
            "capacity": int(i64[2]), "max_tiles": int(i64[3]), "tile": int(i32[8]),
            "bs": int(i32[9]), "lanes": int(i32[10]), "groups": int(i32[11]),
            "merges_tmem": int(i32[12]), "merges_ws": int(i32[13])}


def mla_tree_verify_profiled(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask,
                             mask_indptr, qo_indptr, sm_scale, out, lse, workspace, max_q_per_req,
                             events, stream=None):
    """As mla_tree_verify, recording three torch.cuda.Event objects around the planner
    and the split kernel (events[0..2], on ``stream``)."""
    a = _args(q, kv_cache, kv_indices, kv_indptr, out_cache_loc, custom_mask, mask_indptr,
              qo_indptr, sm_scale, out, lse, workspace, max_q_per_req)
    if len(events) != 3:
        raise MlaTreeVerifyError("need three events")
    for e in events:
        if e.cuda_event == 0:   # created lazily by torch on the first record
            e.record()
    arr = (ctypes.c_void_p * 3)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load().mla_tree_verify_profiled(*a, ctypes.cast(arr, ctypes.c_void_p),
                                           _stream_handle(stream)))


def read_device_status(workspace, stream=None) -> int:
    """Device error bits (DEV_*) of the last call on ``workspace``; synchronises."""
    flags = ctypes.c_uint32(0)
    _check(load().mla_tree_verify_read_device_status(ctypes.c_void_p(workspace.data_ptr()),
                                                     ctypes.byref(flags), _stream_handle(stream)))
    return int(flags.value)


GATHER_BAD_SLOT = 1
GATHER_BAD_ARGS = 2


def kv_gather(kv_cache, kv_indices, kv_indptr, dst, dst_slot0, new_indices, status,
              num_slots=None, stream=None):
    """Enqueues the KV gather-copy (mla_tree_verify_kv_gather in include/mla_tree_verify.h):
    dst row j = kv_cache row kv_indices[kv_indptr[0] + j], new_indices[i] = dst_slot0 +
    i - kv_indptr[0].  ``status`` is a zeroed int32 CUDA tensor of one element that the
    kernel ORs GATHER_BAD_SLOT / GATHER_BAD_ARGS into.  ``num_slots`` (default: rows of
    kv_cache) bounds the valid source slots.  Nothing is synchronised."""
    import torch
    checks = [(kv_cache, torch.bfloat16, 2), (kv_indices, torch.int32, 1),
              (kv_indptr, torch.int32, 1), (dst, torch.bfloat16, 2),
              (new_indices, torch.int32, 1), (status, torch.int32, 1)]
    for t, dt, nd in checks:
        if t.dtype != dt or t.dim() != nd or not t.is_contiguous() or not t.is_cuda:
            raise MlaTreeVerifyError(f"expected a contiguous CUDA {dt} tensor with {nd} dims, "
                                     f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    if kv_cache.shape[1] != D_QK or dst.shape[1] != D_QK:
        raise MlaTreeVerifyError("kv_cache and dst must be [rows, 576]")
    if new_indices.numel() < kv_indices.numel() or status.numel() < 1:
        raise MlaTreeVerifyError("new_indices must be as long as kv_indices; status one word")
    _check(load().mla_tree_verify_kv_gather(
        kv_cache.data_ptr(), int(kv_cache.shape[0] if num_slots is None else num_slots),
        kv_indices.data_ptr(), kv_indices.numel(), kv_indptr.data_ptr(), kv_indptr.shape[0] - 1,
        dst.data_ptr(),
        dst.shape[0], int(dst_slot0), new_indices.data_ptr(), status.data_ptr(),
        _stream_handle(stream)))


CONV1D_PAD_SLOT = -1
CONV1D_BAD_SLOT = 1
CONV1D_BAD_ACCEPT = 2
CONV1D_DTYPE_BF16 = 0
CONV1D_DTYPE_F32 = 1
_CONV1D_ERR = {-1: "a required pointer is NULL", -3: "a size is out of range",
               -4: "a pointer is misaligned", -7: "the launch failed"}


def conv1d_update(x, conv_state, weight, bias, slots, num_accept, window, out, status,
                  silu=True, stream=None):
    """Enqueues the conv-state update of a chain verify with a deduplicated window
    (causal_conv1d_update_dedup_ex in include/causal_conv1d_dedup.h).  CUDA tensors: x and
    out [bs, T, dim], weight [dim, 4] and bias [dim] or None, contiguous, all bf16 or all
    fp32; conv_state [num_slots, dim, state_len] and window [num_slots, dim, T + 2], both
    bf16 or both fp32, any positive strides (a transposed view of the window is fine);
    int32: slots [bs] (CONV1D_PAD_SLOT for a padded row), num_accept [bs] or None, status
    one zeroed word that the kernel ORs CONV1D_BAD_SLOT / CONV1D_BAD_ACCEPT into.  Nothing
    is synchronised."""
    import torch
    codes = {torch.bfloat16: CONV1D_DTYPE_BF16, torch.float32: CONV1D_DTYPE_F32}
    if x.dtype not in codes or conv_state.dtype not in codes:
        raise MlaTreeVerifyError(f"conv1d_update: x and conv_state must be bf16 or fp32, got "
                                 f"{x.dtype} and {conv_state.dtype}")
    checks = [(x, x.dtype, 3, True), (weight, x.dtype, 2, True), (out, x.dtype, 3, True),
              (conv_state, conv_state.dtype, 3, False), (window, conv_state.dtype, 3, False),
              (slots, torch.int32, 1, True), (status, torch.int32, 1, True)]
    if bias is not None:
        checks.append((bias, x.dtype, 1, True))
    if num_accept is not None:
        checks.append((num_accept, torch.int32, 1, True))
    for t, dt, nd, contig in checks:
        if (t.dtype != dt or t.dim() != nd or (contig and not t.is_contiguous()) or not t.is_cuda
                or min(t.stride(), default=1) < 1):
            raise MlaTreeVerifyError(f"expected a CUDA {dt} tensor with {nd} dims"
                                     f"{' (contiguous)' if contig else ''}, got {t.dtype} "
                                     f"{tuple(t.shape)} strides {t.stride()} on {t.device}")
    bs, T, dim = x.shape
    num_slots, _, state_len = conv_state.shape
    if (tuple(out.shape) != (bs, T, dim) or tuple(conv_state.shape[1:2]) != (dim,)
            or tuple(weight.shape) != (dim, 4) or tuple(window.shape) != (num_slots, dim, T + 2)
            or slots.numel() != bs or (bias is not None and bias.numel() != dim)
            or (num_accept is not None and num_accept.numel() != bs)):
        raise MlaTreeVerifyError("conv1d_update: inconsistent shapes")
    ss = (ctypes.c_int64 * 3)(*conv_state.stride())
    ws = (ctypes.c_int64 * 3)(*window.stride())
    rc = load().causal_conv1d_update_dedup_ex(
        x.data_ptr(), conv_state.data_ptr(), weight.data_ptr(),
        None if bias is None else bias.data_ptr(), slots.data_ptr(),
        None if num_accept is None else num_accept.data_ptr(), window.data_ptr(),
        out.data_ptr(), status.data_ptr(), bs, T, dim, state_len, num_slots, int(bool(silu)),
        codes[x.dtype], codes[conv_state.dtype], ctypes.cast(ss, ctypes.c_void_p),
        ctypes.cast(ws, ctypes.c_void_p), _stream_handle(stream))
    if rc != 0:
        raise MlaTreeVerifyError(f"causal_conv1d_update_dedup_ex status {rc}: "
                                 f"{_CONV1D_ERR.get(rc, 'unknown')}")
