"""Helpers for the GPU tests: move a workload to the device and call the library."""
import numpy as np
import torch

import mla_tree_verify_gb300 as mtv
from mla_tree_verify_gb300 import workloads as W

OUT_RTOL = 1e-2   # |out - ref| <= 1e-2 * (1 + |ref|)
LSE_ATOL = 1e-3   # |lse - ref| <= 1e-3


def to_device(wl, device="cuda"):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)
    d = {
        "q": t(wl.q.view(np.int16), torch.int16).view(torch.bfloat16),
        "kv_cache": t(wl.kv_cache.view(np.int16), torch.int16).view(torch.bfloat16),
        "kv_indices": t(wl.kv_indices, torch.int32),
        "kv_indptr": t(wl.kv_indptr, torch.int32),
        "out_cache_loc": t(wl.out_cache_loc, torch.int64),
        "custom_mask": t(wl.custom_mask, torch.uint8),
        "mask_indptr": t(wl.mask_indptr, torch.int64),
        "qo_indptr": t(wl.qo_indptr, torch.int64),
    }
    return d


def alloc_outputs(wl, max_q_per_req=None, device="cuda"):
    mq = max_q_per_req or max(1, wl.max_q_per_req)
    out = torch.full((wl.total_q, wl.num_heads, W.D_V), float("nan"), dtype=torch.bfloat16,
                     device=device)
    lse = torch.full((wl.total_q, wl.num_heads), float("nan"), dtype=torch.float32, device=device)
    ws = torch.empty(mtv.workspace_bytes(wl.bs, mq, wl.num_heads), dtype=torch.uint8,
                     device=device)
    return out, lse, ws, mq


def run(wl, d=None, max_q_per_req=None, sm_scale=None):
    d = d or to_device(wl)
    out, lse, ws, mq = alloc_outputs(wl, max_q_per_req)
    mtv.mla_tree_verify(d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                        d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], d["qo_indptr"],
                        wl.sm_scale if sm_scale is None else sm_scale, out, lse, ws, mq)
    torch.cuda.synchronize()
    return out, lse, ws


def check_rows(out, lse, ref_out, ref_lse, rows):
    """out/lse: device tensors [total_q, H, 512] / [total_q, H]; rows: [n, 2] (row, head);
    ref_out [n, 512] fp64, ref_lse [n]."""
    rows = np.asarray(rows).reshape(-1, 2)
    r = torch.from_numpy(rows[:, 0]).to(out.device)
    h = torch.from_numpy(rows[:, 1]).to(out.device)
    got = out[r, h].float().cpu().numpy().astype(np.float64)
    got_lse = lse[r, h].cpu().numpy().astype(np.float64)
    err = np.abs(got - ref_out) / (1.0 + np.abs(ref_out))
    finite = np.isfinite(ref_lse)
    lse_err = np.where(finite, np.abs(got_lse - np.where(finite, ref_lse, 0.0)), 0.0)
    assert np.all(got_lse[~finite] == -np.inf), "rows with no visible key must give lse=-inf"
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err.max() <= OUT_RTOL, f"max out error {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert lse_err.max() <= LSE_ATOL, f"max lse error {lse_err.max():.3e}"
    return float(err.max()), float(lse_err.max())


def all_rows(wl):
    r, h = np.meshgrid(np.arange(wl.total_q), np.arange(wl.num_heads), indexing="ij")
    return np.stack([r.reshape(-1), h.reshape(-1)], axis=1)


def sample_rows(wl, n, seed=0):
    """n (row, head) pairs: every request's first and last draft, plus random ones."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(wl.bs):
        q0, q1 = int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1])
        if q1 > q0:
            rows.append((q0, int(rng.integers(0, wl.num_heads))))
            rows.append((q1 - 1, int(rng.integers(0, wl.num_heads))))
    extra = max(0, n - len(rows))
    rows += list(zip(rng.integers(0, wl.total_q, extra), rng.integers(0, wl.num_heads, extra)))
    return np.array(rows[:max(n, len(rows))], dtype=np.int64)
