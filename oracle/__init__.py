"""fp64 CPU oracle for MLA tree-verify attention (Python side).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it; the product library never imports it.

The arithmetic lives in ``mla_oracle.c`` (plain fp64 loops over the definition of
masked verify attention; see its header for the cited passages).  This module builds
that file with gcc, loads it with ctypes and passes numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

D_QK = 576
D_V = 512


class _Inputs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("kv", ctypes.c_void_p),
        ("kv_indices", ctypes.c_void_p),
        ("kv_indptr", ctypes.c_void_p),
        ("out_cache_loc", ctypes.c_void_p),
        ("custom_mask", ctypes.c_void_p),
        ("mask_indptr", ctypes.c_void_p),
        ("qo_indptr", ctypes.c_void_p),
        ("bs", ctypes.c_int64),
        ("num_heads", ctypes.c_int64),
        ("num_slots", ctypes.c_int64),
        ("sm_scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compiles mla_oracle.c into a shared library (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp,
                        _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def load_library(path: str):
    """Loads an oracle shared library built from mla_oracle.c (or a variant of it)."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(_Inputs)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.mla_oracle_partial.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, dp, dp, dp]
    lib.mla_oracle_partial.restype = ctypes.c_int
    lib.mla_oracle_combine.argtypes = [ctypes.c_int64, dp, dp, dp, dp, dp]
    lib.mla_oracle_combine.restype = None
    lib.mla_oracle_attend.argtypes = [P, ctypes.c_void_p, ctypes.c_int64, dp, dp, ctypes.c_int]
    lib.mla_oracle_attend.restype = ctypes.c_int
    lib.mla_oracle_enumerate.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p]
    lib.mla_oracle_enumerate.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Oracle:
    """Binds one workload's arrays (kept alive here) to the C oracle."""

    def __init__(self, wl, sm_scale: float | None = None, lib=None):
        self._keep = [
            np.ascontiguousarray(wl.q, dtype=np.uint16),
            np.ascontiguousarray(wl.kv_cache, dtype=np.uint16),
            np.ascontiguousarray(wl.kv_indices, dtype=np.int32),
            np.ascontiguousarray(wl.kv_indptr, dtype=np.int32),
            np.ascontiguousarray(wl.out_cache_loc, dtype=np.int64),
            np.ascontiguousarray(wl.custom_mask, dtype=np.uint8),
            np.ascontiguousarray(wl.mask_indptr, dtype=np.int64),
            np.ascontiguousarray(wl.qo_indptr, dtype=np.int64),
        ]
        k = self._keep
        self.bs = int(k[3].shape[0] - 1)
        self.num_heads = int(wl.q.shape[1])
        self.total_q = int(k[7][-1])
        self.inputs = _Inputs(
            k[0].ctypes.data, k[1].ctypes.data, k[2].ctypes.data, k[3].ctypes.data,
            k[4].ctypes.data, k[5].ctypes.data, k[6].ctypes.data, k[7].ctypes.data,
            self.bs, self.num_heads, int(wl.kv_cache.shape[0]),
            float(wl.sm_scale if sm_scale is None else sm_scale))
        self.lib = lib if lib is not None else _load()

    def attend(self, rows: np.ndarray | None = None, threads: int | None = None):
        """(out [n,512], lse [n]) for (row, head) pairs ``rows`` [n,2], or for every
        pair in (row, head) order when rows is None."""
        threads = threads or os.cpu_count() or 1
        if rows is None:
            n = self.total_q * self.num_heads
            rp = None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
            n = rows.shape[0]
            rp = rows.ctypes.data
        out = np.zeros((n, D_V), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        st = self.lib.mla_oracle_attend(ctypes.byref(self.inputs), rp, n, _dptr(out), _dptr(lse),
                                        threads)
        if st != 0:
            raise RuntimeError(f"oracle status {st}")
        return out, lse

    def partial(self, r: int, h: int, c0: int, c1: int):
        o = np.zeros(D_V, dtype=np.float64)
        m = np.zeros(1, dtype=np.float64)
        l = np.zeros(1, dtype=np.float64)
        st = self.lib.mla_oracle_partial(ctypes.byref(self.inputs), r, h, c0, c1, _dptr(o),
                                         _dptr(m), _dptr(l))
        if st != 0:
            raise RuntimeError(f"oracle status {st}")
        return float(m[0]), float(l[0]), o

    def enumerate(self):
        """(slots int64 [sum_b L_b], vis uint8 [mask length])."""
        L = np.diff(self._keep[3].astype(np.int64)) + np.diff(self._keep[7])
        slots = np.zeros(int(L.sum()), dtype=np.int64)
        vis = np.zeros(self._keep[5].shape[0], dtype=np.uint8)
        st = self.lib.mla_oracle_enumerate(ctypes.byref(self.inputs), slots.ctypes.data,
                                           vis.ctypes.data)
        if st != 0:
            raise RuntimeError(f"oracle status {st}")
        return slots, vis


def kv_gather(kv, kv_indices, kv_indptr, dst_rows, dst_slot0, lib=None):
    """The KV gather-copy (see mla_oracle_kv_gather in mla_oracle.c): returns
    (dst uint16 [dst_rows, 576], new_indices int32 like kv_indices, bad entries)."""
    lib = lib if lib is not None else _load()
    kv = np.ascontiguousarray(kv, dtype=np.uint16)
    idx = np.ascontiguousarray(kv_indices, dtype=np.int32)
    ptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    dst = np.zeros((dst_rows, 576), dtype=np.uint16)
    new = np.zeros_like(idx)
    lib.mla_oracle_kv_gather.restype = ctypes.c_int64
    lib.mla_oracle_kv_gather.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    bad = lib.mla_oracle_kv_gather(kv.ctypes.data, kv.shape[0], idx.ctypes.data, ptr.ctypes.data,
                                   ptr.shape[0] - 1, dst.ctypes.data, dst_rows, dst_slot0,
                                   new.ctypes.data)
    if bad < 0:
        raise ValueError("kv_gather: bad arguments")
    return dst, new, int(bad)


def combine(m, l, o, lib=None):
    """Merges partials (m [n], l [n], o [n,512]) -> (out [512], lse)."""
    lib = lib if lib is not None else _load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64).reshape(-1, D_V)
    out = np.zeros(D_V, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.mla_oracle_combine(m.shape[0], _dptr(m), _dptr(l), _dptr(o), _dptr(out), _dptr(lse))
    return out, float(lse[0])
