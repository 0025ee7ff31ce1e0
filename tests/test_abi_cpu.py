"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports every
function that include/*.h declares, and rejects bad arguments on the host before it
touches a device."""
import ctypes
import glob
import os
import re

import pytest

from mla_tree_verify_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:int|int32_t|size_t|void|const\s+char\s*\*)\s*(\w+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("mla_tree_verify", "mla_tree_verify_workspace_bytes", "mla_tree_verify_debug",
              "mla_tree_verify_prepare", "mla_tree_verify_read_device_status",
              "mla_tree_verify_status_string", "mla_tree_verify_split_grid",
              "mla_tree_verify_kv_gather", "causal_conv1d_update_dedup",
              "causal_conv1d_update_dedup_ex"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        s = lib.mla_tree_verify_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.mla_tree_verify_status_string(12345).decode() == "unknown status"


def _call(lib, **over):
    a = dict(q=16, kv=16, kvi=16, kvp=16, ocl=16, mask=16, mip=16, qop=16, scale=0.1, out=16,
             lse=16, ws=256, wsb=1 << 30, bs=1, mq=4, heads=64, slots=10, total_q=4, nkvi=3,
             mlen=28)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.mla_tree_verify(vp(a["q"]), vp(a["kv"]), vp(a["kvi"]), vp(a["kvp"]), vp(a["ocl"]),
                               vp(a["mask"]), vp(a["mip"]), vp(a["qop"]), ctypes.c_float(a["scale"]),
                               vp(a["out"]), vp(a["lse"]), vp(a["ws"]), a["wsb"], a["bs"], a["mq"],
                               a["heads"], a["slots"], a["total_q"], a["nkvi"], a["mlen"], vp(0))


def test_host_argument_checks(lib):
    # these are rejected before any device query or launch (the pointers are never used)
    assert _call(lib, heads=32) == -2
    assert _call(lib, bs=0) == -3
    assert _call(lib, mq=0) == -3
    assert _call(lib, mq=5000) == -3
    assert _call(lib, q=0) == -1
    assert _call(lib, ws=0) == -1
    assert _call(lib, kvi=0) == -1              # num_kv_indices > 0 needs kv_indices
    assert _call(lib, kvi=0, nkvi=0) != -1      # ... but not when it is empty
    assert _call(lib, scale=float("inf")) == -8
    assert _call(lib, q=8) == -4
    assert _call(lib, ws=512 + 16) == -4


def test_no_device_here(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.mla_tree_verify_workspace_bytes(8, 16, 64) == 0
    assert _call(lib) == -7
    assert lib.mla_tree_verify_prepare() == -7


def test_workspace_query_rejects_bad_shapes(lib):
    assert lib.mla_tree_verify_workspace_bytes(8, 16, 32) == 0
    assert lib.mla_tree_verify_workspace_bytes(0, 16, 64) == 0


def _gather(lib, **over):
    a = dict(kv=16, slots=10, kvi=16, nkvi=8, kvp=16, bs=1, dst=16, rows=8, slot0=0, new=16,
             st=16)
    a.update(over)
    vp = ctypes.c_void_p
    return lib.mla_tree_verify_kv_gather(vp(a["kv"]), a["slots"], vp(a["kvi"]), a["nkvi"],
                                         vp(a["kvp"]), a["bs"], vp(a["dst"]), a["rows"],
                                         a["slot0"], vp(a["new"]), vp(a["st"]), vp(0))


def test_kv_gather_host_argument_checks(lib):
    lib.mla_tree_verify_kv_gather.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    lib.mla_tree_verify_kv_gather.restype = ctypes.c_int
    assert _gather(lib, kv=0) == -1
    assert _gather(lib, dst=0) == -1
    assert _gather(lib, st=0) == -1
    assert _gather(lib, bs=0) == -3
    assert _gather(lib, slots=0) == -3
    assert _gather(lib, nkvi=-1) == -3
    assert _gather(lib, rows=-1) == -3
    assert _gather(lib, slot0=-1) == -3
    assert _gather(lib, slot0=(1 << 31) - 4, rows=8) == -3     # new indices past INT32_MAX
    assert _gather(lib, kv=8) == -4
    assert _gather(lib, dst=24) == -4
    assert _gather(lib, kvi=18) == -4


def test_kv_gather_needs_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _gather(lib) == -7


def _conv(lib, x=16, st=32, w=48, bias=64, slots=80, acc=0, win=96, out=112, status=128, bs=2,
          T=8, dim=16, state_len=3, num_slots=4, silu=1):
    return lib.causal_conv1d_update_dedup(x, st, w, bias, slots, acc, win, out, status, bs, T,
                                          dim, state_len, num_slots, silu, None)


def test_conv1d_host_argument_checks(lib):
    """Null pointers, sizes and alignment are rejected before any device call (the fake
    addresses are never dereferenced)."""
    for kw in ("x", "st", "w", "slots", "win", "out", "status"):
        assert _conv(lib, **{kw: 0}) == -1, kw
    assert _conv(lib, bias=0) != -1 and _conv(lib, acc=0) != -1      # optional inputs
    for kw, v in (("bs", 0), ("T", 0), ("T", 17), ("dim", 0), ("dim", 12), ("state_len", 2),
                  ("state_len", 33), ("num_slots", 0), ("num_slots", 1 << 31)):
        assert _conv(lib, **{kw: v}) == -3, (kw, v)
    for kw in ("x", "st", "w", "bias", "win", "out"):
        assert _conv(lib, **{kw: 24}) == -4, kw


def test_conv1d_needs_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _conv(lib) == -7


def _conv_ex(lib, x=16, st=32, w=48, bias=64, slots=80, acc=0, win=96, out=112, status=128, bs=2,
             T=8, dim=16, state_len=3, num_slots=4, silu=1, xd=0, sd=0, ss=None, ws=None):
    arr = lambda v: None if v is None else ctypes.cast((ctypes.c_int64 * 3)(*v), ctypes.c_void_p)
    return lib.causal_conv1d_update_dedup_ex(x, st, w, bias, slots, acc, win, out, status, bs, T,
                                             dim, state_len, num_slots, silu, xd, sd, arr(ss),
                                             arr(ws), None)


def test_conv1d_ex_host_argument_checks(lib):
    """The general entry: type codes, strides and element alignment are checked on the host;
    any channel count and 2- or 4-byte aligned pointers pass to the launch (which needs a
    device)."""
    for kw in ("x", "st", "w", "slots", "win", "out", "status"):
        assert _conv_ex(lib, **{kw: 0}) == -1, kw
    for kw, v in (("bs", 0), ("T", 17), ("dim", 0), ("state_len", 2), ("num_slots", 0),
                  ("xd", 2), ("sd", -1), ("ss", (0, 3, 1)), ("ws", (10, -1, 1))):
        assert _conv_ex(lib, **{kw: v}) == -3, (kw, v)
    for kw in ("x", "w", "bias", "out"):
        assert _conv_ex(lib, **{kw: 17}) == -4, kw               # bf16: 2-byte alignment
        assert _conv_ex(lib, xd=1, **{kw: 18}) == -4, kw         # fp32: 4-byte alignment
    for kw in ("st", "win"):
        assert _conv_ex(lib, **{kw: 17}) == -4, kw
        assert _conv_ex(lib, sd=1, **{kw: 18}) == -4, kw
    import torch
    if torch.cuda.is_available():
        return
    for kw in ({"dim": 13}, {"x": 18}, {"xd": 1}, {"sd": 1}, {"ws": (10, 1, 16 * 4)},
               {"ss": (3, 1, 16)}):
        assert _conv_ex(lib, **kw) == -7, kw
