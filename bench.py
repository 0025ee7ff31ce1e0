#!/usr/bin/env python
"""Benchmark of MLA tree-verify attention on one GB300 (or N replicas).

Default workload (the largest single-GPU config): bs=64 requests, 64 heads, q/kv dim 576
(V = first 512), bf16 N(0,1)*0.5 q and kv with 1% of rows x8 (outliers); prefix lengths
uniform in [8192, 65536] scattered page_size=1 over a 4,194,304-slot pool; per request
T in {1, 4, 8, 16} draft tokens in a random tree (parent of node i uniform in [0, i));
mask = ancestor-or-self; sm_scale = 1/sqrt(192); NSPLIT = 64; calls replayed from a
CUDA graph.

One step = one call of the C-ABI entry point (planner + split kernel) on inputs already
resident in HBM; L2 is flushed (256 MiB write) between timed steps, outside the timed
events.  Prints one JSON line, which also holds every verify config (1-5) measured one
after another under "per_config".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference] [--shape k]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call + KV HBM GB/s (% of GB300 roofline) for MLA tree verify at bs×T×ctx"
UNIT = "us/call"
FLOPS_PER_PAIR = 2 * 576 + 2 * 512   # one visible (query row, key) pair, per head
_EXTERNAL_EVENTS = True               # torch.cuda.Event(external=True) available


def _timing_event():
    """A timing event whose records inside a graph capture stay readable after replay."""
    global _EXTERNAL_EVENTS
    import torch
    if _EXTERNAL_EVENTS:
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            _EXTERNAL_EVENTS = False
    return torch.cuda.Event(enable_timing=True)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def workload_counts(wl):
    pairs = wl.visible_pairs()               # visible (token, key) pairs, per head
    flops = pairs * wl.num_heads * FLOPS_PER_PAIR
    return {"kv_bytes": wl.kv_bytes(), "flops": flops, "visible_pairs": pairs,
            "qk_pairs_total": wl.total_q * wl.num_heads}


def config_of(wl, name):
    P = wl.prefix_lens
    return {"workload": name, "bs": wl.bs, "heads": wl.num_heads, "d_qk": 576, "d_v": 512,
            "T_per_request": sorted(set(int(x) for x in wl.draft_lens)),
            "prefix_min": int(P.min()), "prefix_max": int(P.max()),
            "prefix_mean": float(P.mean()), "pool_slots": wl.num_slots, "nsplit": 64,
            "l2": "flushed by a 256 MiB write between timed steps (outside the events)"}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# The sources each profiled kernel is built from: a committed ncu summary records their
# hash, and its counters are reported only while the hash still matches.
KERNEL_SOURCES = {
    "split": ["mtv_split_tc.cu", "mtv_plan.cu", "mtv_api.cu", "mtv_common.cuh", "mtv_ptx.cuh"],
    "kv_gather": ["mtv_kv_gather.cu", "mtv_api.cu", "mtv_common.cuh"],
    "conv1d": ["mtv_conv1d.cu"],
    "conv1d_general": ["mtv_conv1d_general.cu"],
}


def kernel_sha(kernel):
    from mla_tree_verify_gb300 import build as b
    return source_sha([os.path.join(b.CSRC, f) for f in KERNEL_SOURCES[kernel]])


def source_sha(paths):
    """Hash of the sources' code: comments and whitespace are left out, so that editing a
    comment does not mark a profile of the same code as stale."""
    import re
    h = hashlib.sha256()
    for p in paths:
        with open(p) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


# workload name -> committed ncu summary of the split kernel on it (or on a smaller draw
# of the same distribution, whose DRAM bytes per algorithmic KV byte are scaled)
SPLIT_PROFILES = {
    "bs8_P1k-4k_T16_tree_pool65536": "split_kernel_bs8_T16_P1k-4k.md",
    "bs8_P1k-4k_T16_tree_pool65536_contiguous": "split_kernel_bs8_T16_P1k-4k_contiguous.md",
    "bs64_P8k-64k_Tmix_tree_outliers_pool4M": "split_kernel_bs64_P8k-64k_Tmix.md",
    "bs32_P512-32k_logU_T8_chain_pool1M": "split_kernel_bs32_P512-32k_T8.md",
}


def split_kernel_traffic(name, kv_bytes=None):
    """DRAM bytes per split-kernel launch on workload `name` from the committed ncu
    summary, if there is one and it was taken on the current kernel sources (else None).
    A summary taken on a smaller draw of the workload's distribution gives DRAM bytes
    per algorithmic KV byte, scaled here to the workload's KV bytes."""
    import re
    if name not in SPLIT_PROFILES:
        return None
    path = os.path.join(ROOT, "profiles", SPLIT_PROFILES[name])
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"csrc_sha: ([0-9a-f]+)", text)
    if not sha or sha.group(1) != kernel_sha("split"):
        return None
    val = re.search(r"dram_bytes_per_launch: (\d+)", text)
    if val:
        return int(val.group(1))
    ratio = re.search(r"dram_bytes_per_kv_byte: ([0-9.]+)", text)
    if ratio and kv_bytes:
        return int(float(ratio.group(1)) * kv_bytes)
    return None


def cpu_baseline(wl, seconds, seed=0):
    """Times the fp64 oracle on a uniform sample of (row, head) pairs on all host cores
    and scales to one full call."""
    import numpy as np
    import oracle
    orc = oracle.Oracle(wl)
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    total_pairs = wl.total_q * wl.num_heads
    n, spent, done = max(threads, 8), 0.0, 0
    while spent < seconds and done < total_pairs:
        rows = np.stack([rng.integers(0, wl.total_q, n), rng.integers(0, wl.num_heads, n)], 1)
        t0 = time.perf_counter()
        orc.attend(rows, threads=threads)
        dt = time.perf_counter() - t0
        spent += dt
        done += n
        n = min(4 * n, max(threads, int(n * max(1.0, (seconds - spent) / max(dt, 1e-3)))))
    us = spent / done * total_pairs * 1e6
    return {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} (row, head) pairs drawn uniformly from the {total_pairs} of the "
                      f"workload, fp64 C oracle on {threads} OpenMP threads, {spent:.1f} s, "
                      f"scaled by {total_pairs}/{done}"}


def max_over_ranks(value, device=None):
    """The largest value over the ranks of the default process group (the value itself
    when there is none): the job takes as long as its slowest replica."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    x = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def whole_job_us_per_call(t_max_ms, steps, world):
    """Whole-job µs per call for `world` replicas that each made `steps` calls within
    t_max_ms milliseconds."""
    return t_max_ms * 1e3 / (steps * world)


def run_reference(args, wl, name):
    """The oracle as it stands, on the host cores: each step times a sample of (row, head)
    pairs drawn uniformly from the workload and scales it to one full call.  A step takes
    64 pairs per core, fewer only where that would make the whole run (warm-up and timed
    steps) exceed about four minutes."""
    import numpy as np
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    orc = oracle.Oracle(wl)
    threads = os.cpu_count() or 1
    total_pairs = wl.total_q * wl.num_heads
    rng = np.random.default_rng(1)

    def timed(n):
        rows = np.stack([rng.integers(0, wl.total_q, n), rng.integers(0, wl.num_heads, n)], 1)
        t0 = time.perf_counter()
        orc.attend(rows, threads=threads)
        return time.perf_counter() - t0

    # calibration: seconds per pair with every core busy
    per_pair = timed(4 * threads) / (4 * threads)
    budget_s = 240.0 / (args.steps + args.warmup)
    n = int(min(64 * threads, max(threads, budget_s / max(per_pair, 1e-9))))
    n = max(threads, n - n % threads)
    walls = []

    def step():
        dt = timed(n)
        walls.append(dt)
        return dt / n * total_pairs * 1e6

    for _ in range(args.warmup):
        step()
    t = [step() for _ in range(args.steps)]
    v = statistics.mean(t)
    sample = (f"{n} (row, head) pairs per step ({n // threads} per core) drawn uniformly from the "
              f"{total_pairs} of one call, fp64 C oracle on {threads} OpenMP threads; each step's "
              f"time is scaled by {total_pairs}/{n} to one call (an extrapolation of a sample)")
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": config_of(wl, name),
            "extrapolated_from_sample": True,
            "sample_wall_s_per_step": statistics.mean(walls[args.warmup:]),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def kv_gather_traffic():
    """DRAM bytes per gather launch (bench workload) from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    import re
    path = os.path.join(ROOT, "profiles", "kv_gather_bs32_P512-32k.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"csrc_sha: ([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch: (\d+)", text)
    if not sha or not val:
        return None
    if sha.group(1) != kernel_sha("kv_gather"):
        return None
    return int(val.group(1))


def bench_kv_gather(args, wl, name):
    """The KV gather-copy of the shape's prefix rows into a contiguous destination: GB/s
    of algorithmic traffic (rows read and written once, indices read and rewritten),
    against the measured HBM copy peak; the oracle's gather timed on the host."""
    import numpy as np
    import torch
    import mla_tree_verify_gb300 as mtv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    kv = torch.from_numpy(wl.kv_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    idx_h = np.ascontiguousarray(wl.kv_indices, dtype=np.int32)
    ptr_h = np.ascontiguousarray(wl.kv_indptr, dtype=np.int32)
    idx = torch.from_numpy(idx_h).to(dev)
    ptr = torch.from_numpy(ptr_h).to(dev)
    n = idx.numel()
    dst = torch.empty((n, 576), dtype=torch.bfloat16, device=dev)
    new = torch.empty_like(idx)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    mtv.prepare()
    for _ in range(args.warmup):
        flush.zero_()
        mtv.kv_gather(kv, idx, ptr, dst, 0, new, status)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("gather status flags set")
    K = args.steps
    # Between timed steps L2 must not hold the rows: when the rows read and written are
    # larger than L2 (129 MB) the copy itself evicts them; otherwise a 256 MiB write
    # flushes L2 (its dirty lines are then written back during the next step).
    big = n * 1152 * 2 > 129e6
    stream = torch.cuda.Stream()
    graphs, left = [], K
    _timing_event()
    while left > 0:
        m = min(50, left)
        ev = [[_timing_event(), _timing_event()] for _ in range(m)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for a, b in ev:
                a.record()
                b.record()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for a, b in ev:
                    if not big:
                        flush.zero_()
                    a.record(stream)
                    mtv.kv_gather(kv, idx, ptr, dst, 0, new, status, stream=stream)
                    b.record(stream)
        graphs.append((g, ev))
        left -= m
    for g, _ in graphs:
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t = []
    for g, ev in graphs:
        g.replay()
        torch.cuda.synchronize()
        t += [a.elapsed_time(b) for a, b in ev]
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError("gather status flags set")
    us = statistics.mean(t) * 1e3
    nbytes = n * 1152 * 2 + n * 4 * 2 + ptr.numel() * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    hbm_gbs, _, src = peaks()
    # end to end: the index arrays come from pinned host memory, the status word goes back
    pin_idx = torch.from_numpy(idx_h).pin_memory()
    pin_ptr = torch.from_numpy(ptr_h).pin_memory()
    st_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    e2e = []
    for i in range(args.e2e_steps + 3):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        idx.copy_(pin_idx, non_blocking=True)
        ptr.copy_(pin_ptr, non_blocking=True)
        mtv.kv_gather(kv, idx, ptr, dst, 0, new, status)
        st_h.copy_(status, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            e2e.append(e0.elapsed_time(e1))
    e2e_us = statistics.mean(e2e) * 1e3
    line = {
        "metric": "KV gather-copy (defragmentation step) GB/s", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": us * 1e-3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name + "_prefix_rows", "rows": n, "row_bytes": 1152,
                   "l2": ("inputs larger than L2 (rows read + written), no flush" if big else
                          "flushed by a 256 MiB write between timed steps (outside the events)")},
        "us_per_call": us,
        "roofline": {"bound": "hbm", "kernel": "kv_gather", "achieved": gbs, "peak": hbm_gbs,
                     "unit": "GB/s", "frac": gbs / hbm_gbs,
                     "peak_source": f"{src} HBM copy (burst)",
                     "traffic": (kv_gather_traffic()
                                 if name == "bs32_P512-32k_logU_T8_chain_pool1M" else None),
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": e2e_us, "unit": "us/call",
                "h2d_bytes_per_step": (idx_h.nbytes + ptr_h.nbytes), "d2h_bytes_per_step": 4},
        "gpu_launches": K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle     # the CPU baseline leg: the oracle's gather, as it stands
        kvh = np.ascontiguousarray(wl.kv_cache, dtype=np.uint16)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0) or reps == 0:
            oracle.kv_gather(kvh, idx_h, ptr_h, n, 0)
            reps += 1
        cpu_s = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": nbytes / cpu_s / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"the whole gather ({n} rows), {reps} runs, "
                                          "single-threaded C loop"}
    print(json.dumps(line), flush=True)


# Kernel time per call of the deduplicated-window tile store, GB300, dim 10240, K 4, bf16,
# CUDA graph: the pull request "jianc99/sglang#1", section "Benchmarking and Profiling"
# (its "after" column), keyed by (bs, T).
CONV1D_PUBLISHED_US = {(1, 8): 2.49, (64, 8): 9.96, (128, 8): 17.55, (128, 16): 39.10}


def conv1d_traffic(kernel="conv1d", profile="conv1d_dedup_bs128_T8_dim10240.md"):
    """DRAM bytes per conv-update launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    import re
    path = os.path.join(ROOT, "profiles", profile)
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"csrc_sha: ([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch: (\d+)", text)
    if not sha or not val:
        return None
    return int(val.group(1)) if sha.group(1) == kernel_sha(kernel) else None


def bench_defrag_verify(args, wl, name):
    """Each step defragments the shape's prefix rows (the KV gather-copy into free slots at
    the end of the pool, indices rewritten) and then runs verify through the new indices,
    so that full prefix tiles load as TMA tile copies.  The two calls are timed together,
    L2 flushed between steps: the cost of defragmenting before every verify."""
    import numpy as np
    import torch
    import mla_tree_verify_gb300 as mtv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dt)
    n = int(wl.kv_indices.shape[0])
    slots = wl.num_slots
    pool = torch.empty((slots + n, 576), dtype=torch.bfloat16, device=dev)
    pool[:slots].copy_(t(wl.kv_cache.view(np.int16), torch.bfloat16))
    q = t(wl.q.view(np.int16), torch.bfloat16)
    idx, ptr = t(wl.kv_indices, torch.int32), t(wl.kv_indptr, torch.int32)
    ocl, msk = t(wl.out_cache_loc, torch.int64), t(wl.custom_mask, torch.uint8)
    mptr, qptr = t(wl.mask_indptr, torch.int64), t(wl.qo_indptr, torch.int64)
    new = torch.empty_like(idx)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mq = wl.max_q_per_req
    out = torch.empty((wl.total_q, wl.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.total_q, wl.num_heads), dtype=torch.float32, device=dev)
    ws = torch.empty(mtv.workspace_bytes(wl.bs, mq, wl.num_heads), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    mtv.prepare()

    def step(stream=None):
        mtv.kv_gather(pool, idx, ptr, pool[slots:], slots, new, status, num_slots=slots,
                      stream=stream)
        mtv.mla_tree_verify(q, pool, new, ptr, ocl, msk, mptr, qptr, wl.sm_scale, out, lse, ws,
                            mq, stream=stream)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0 or mtv.read_device_status(ws) != 0:
        raise RuntimeError("status flags set")
    stream = torch.cuda.Stream()
    graphs, left = [], args.steps
    _timing_event()
    while left > 0:
        m = min(50, left)
        ev = [[_timing_event(), _timing_event()] for _ in range(m)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for a, e in ev:
                a.record()
                e.record()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for a, e in ev:
                    flush.zero_()
                    a.record(stream)
                    step(stream)
                    e.record(stream)
        graphs.append((g, ev))
        left -= m
    for g, _ in graphs:
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    times = []
    for g, ev in graphs:
        g.replay()
        torch.cuda.synchronize()
        times += [a.elapsed_time(e) for a, e in ev]
    clk = clocks.stop()
    us = statistics.mean(times) * 1e3
    c = workload_counts(wl)
    hbm_gbs, tc_tflops, src = peaks()
    line = {"metric": "gather-copy + verify, us/call", "value": us, "unit": "us/call",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us * 1e-3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(config_of(wl, name + "_defragmented_each_step")),
            "roofline": {"bound": "tensor", "kernel": "split + gather (call)",
                         "achieved": c["flops"] / (us * 1e-6) / 1e12, "peak": tc_tflops,
                         "unit": "TFLOP/s", "frac": c["flops"] / (us * 1e-6) / 1e12 / tc_tflops,
                         "peak_source": f"{src} bf16 dense (burst)", "traffic": None},
            "gpu_launches": 3 * args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


def run_reference_conv1d(args):
    """The conv-update oracle as it stands, on the host: each step is one whole call on the
    same workload as --kernel conv1d."""
    from mla_tree_verify_gb300 import conv_workloads as CW
    import oracle.conv1d as O
    if int(os.environ.get("RANK", "0")) != 0:
        return
    bs, T = args.conv_bs, args.conv_t
    xd, sd = args.conv_types.split(",")
    c = CW.case(20261300 + bs + T, bs=bs, T=T, dim=CW.BENCH_DIM, x_dtype=xd, state_dtype=sd)
    name = f"conv1d_dedup_bs{bs}_T{T}_dim{CW.BENCH_DIM}_K4"
    if (xd, sd, args.conv_window) != ("bf16", "bf16", "contiguous"):
        name += f"_x{xd}_state{sd}_window{args.conv_window}"

    def step():
        t0 = time.perf_counter()
        O.update(c)
        return (time.perf_counter() - t0) * 1e6
    for _ in range(args.warmup):
        step()
    t = [step() for _ in range(args.steps)]
    v = statistics.mean(t)
    line = {"metric": "conv-state update with a deduplicated window, us/call", "value": v,
            "unit": "us/call", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": v / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": name, "bs": bs, "T": T, "dim": CW.BENCH_DIM,
                       "input_dtype": xd, "state_dtype": sd, "window": args.conv_window},
            "cpu_baseline": {"value": v, "unit": "us/call", "cores": 1, "kind": "oracle",
                             "sample": "the whole call per step, numpy fp64 (one thread)"},
            "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_conv1d(args):
    """The conv-state update of a chain verify with a deduplicated window, at dim 10240:
    µs per call and GB/s of algorithmic bytes against the measured HBM copy peak; the
    fp64 oracle timed on the host."""
    import numpy as np
    import torch
    import mla_tree_verify_gb300 as mtv
    from mla_tree_verify_gb300 import conv_workloads as CW
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    bs, T = args.conv_bs, args.conv_t
    xd, sd = args.conv_types.split(",")
    c = CW.case(20261300 + bs + T, bs=bs, T=T, dim=CW.BENCH_DIM, x_dtype=xd, state_dtype=sd)

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    x, st, w, b = to_dev(c.x), to_dev(c.conv_state), to_dev(c.weight), to_dev(c.bias)
    slots, win, out = to_dev(c.slots), to_dev(c.window), to_dev(c.out)
    if args.conv_window == "transposed":     # the window rows stored column-major over slots
        win_phys = torch.empty((T + 2, c.num_slots, c.dim), dtype=win.dtype, device=dev)
        win_phys.permute(1, 2, 0).copy_(win)
        win = win_phys.permute(1, 2, 0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call(stream=None):
        mtv.conv1d_update(x, st, w, b, slots, None, win, out, status, silu=c.silu, stream=stream)
    def flush_l2():
        # write a buffer larger than L2, then read it, so that the timed call starts with
        # L2 holding none of its data and no dirty lines left to write back
        flush.zero_()
        flush.sum(dtype=torch.int32)
    for _ in range(args.warmup):
        flush_l2()
        call()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("conv1d status flags set")
    K = args.steps
    stream = torch.cuda.Stream()
    graphs, left = [], K
    _timing_event()
    while left > 0:
        m = min(50, left)
        ev = [[_timing_event(), _timing_event()] for _ in range(m)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for a, e in ev:
                a.record()
                e.record()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for a, e in ev:
                    flush_l2()
                    a.record(stream)
                    call(stream)
                    e.record(stream)
        graphs.append((g, ev))
        left -= m
    for g, _ in graphs:
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    times = []
    for g, ev in graphs:
        g.replay()
        torch.cuda.synchronize()
        times += [a.elapsed_time(e) for a, e in ev]
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError("conv1d status flags set")
    us = statistics.mean(times) * 1e3
    # context only: the same call replayed back to back with no flush (inputs partly left
    # in L2 by the previous call), as a graph of 50 calls timed as a whole
    g_warm = torch.cuda.CUDAGraph()
    ew = [_timing_event(), _timing_event()]
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_warm, stream=stream):
            ew[0].record(stream)
            for _ in range(50):
                call(stream)
            ew[1].record(stream)
    warm = []
    for _ in range(5):
        g_warm.replay()
        torch.cuda.synchronize()
        warm.append(ew[0].elapsed_time(ew[1]) * 1e3 / 50)
    us_warm = statistics.median(warm)
    nbytes = c.algorithmic_bytes()
    gbs = nbytes / (us * 1e-6) / 1e9
    hbm_gbs, _, src = peaks()
    # end to end: the step's inputs (x, slots) from pinned host memory, its output back;
    # the conv state pool and the window rows stay resident, as the model's state does
    x_bits = x.view(torch.int16) if x.dtype == torch.bfloat16 else x
    x_h = torch.from_numpy(c.x.view(np.int16) if xd == "bf16" else c.x).pin_memory()
    slots_h = torch.from_numpy(c.slots).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e = []
    for i in range(args.e2e_steps + 3):
        flush_l2()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        x_bits.copy_(x_h, non_blocking=True)
        slots.copy_(slots_h, non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            e2e.append(e0.elapsed_time(e1))
    e2e_us = statistics.mean(e2e) * 1e3
    default = (xd, sd, args.conv_window) == ("bf16", "bf16", "contiguous")
    pub = CONV1D_PUBLISHED_US.get((bs, T)) if default else None
    name = f"conv1d_dedup_bs{bs}_T{T}_dim{CW.BENCH_DIM}_K4"
    if not default:
        name += f"_x{xd}_state{sd}_window{args.conv_window}"
    fast = (xd, sd) == ("bf16", "bf16")    # the 4-channels-a-thread kernel, either window layout
    line = {
        "metric": "conv-state update with a deduplicated window, us/call", "value": us,
        "unit": "us/call", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": us * 1e-3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": (us / pub) if pub else None,
        "dtype": xd if xd == sd else f"{xd} inputs, {sd} state", "data": "synthetic",
        "config": {"workload": name, "bs": bs, "T": T, "dim": CW.BENCH_DIM,
                   "state_len": c.state_len, "silu": c.silu, "input_dtype": xd,
                   "state_dtype": sd, "window": args.conv_window,
                   "l2": "flushed between timed steps (outside the events) by a 256 MiB write "
                         "and a read of the same buffer"},
        "gbs": gbs,
        "us_per_call_back_to_back_no_flush": us_warm,
        "roofline": {"bound": "hbm", "kernel": "conv1d_dedup" if fast else "conv1d_general",
                     "achieved": gbs, "peak": hbm_gbs,
                     "unit": "GB/s", "frac": gbs / hbm_gbs,
                     "peak_source": f"{src} HBM copy (burst)",
                     "traffic": (conv1d_traffic() if default else None if fast else conv1d_traffic(
                         "conv1d_general", "conv1d_general_bs128_T8_dim10240_f32.md")
                         if (xd, sd, args.conv_window) == ("f32", "f32", "contiguous") else None)
                     if (bs, T) == (128, 8) else None,
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": {"value": e2e_us, "unit": "us/call",
                "h2d_bytes_per_step": int(c.x.nbytes + c.slots.nbytes),
                "d2h_bytes_per_step": int(out.numel() * out.element_size())},
        "gpu_launches": K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle.conv1d as O     # the CPU baseline leg: the oracle, as it stands
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < min(args.cpu_seconds, 10.0) or reps == 0:
            O.update(c)
            reps += 1
        cpu_s = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": cpu_s * 1e6, "unit": "us/call", "cores": 1,
                                "kind": "oracle",
                                "sample": f"the whole call, {reps} runs, numpy fp64 (one thread)"}
    print(json.dumps(line), flush=True)



class VerifySetup:
    """One verify workload moved to the device, with its outputs and a workspace, ready
    to be called through the C ABI."""

    DTYPES = {"q": "bfloat16", "kv_cache": "bfloat16", "kv_indices": "int32",
              "kv_indptr": "int32", "out_cache_loc": "int64", "custom_mask": "uint8",
              "mask_indptr": "int64", "qo_indptr": "int64"}

    def __init__(self, wl, dev, lanes=0):
        import numpy as np
        import torch
        import mla_tree_verify_gb300 as mtv
        self.wl, self.dev, self.mtv, self.lanes = wl, dev, mtv, lanes
        self.host = {"q": wl.q.view(np.int16), "kv_cache": wl.kv_cache.view(np.int16),
                     "kv_indices": wl.kv_indices, "kv_indptr": wl.kv_indptr,
                     "out_cache_loc": wl.out_cache_loc, "custom_mask": wl.custom_mask,
                     "mask_indptr": wl.mask_indptr, "qo_indptr": wl.qo_indptr}
        self.d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev).view(
            getattr(torch, self.DTYPES[k])) for k, v in self.host.items()}
        mq = wl.max_q_per_req
        self.out = torch.empty((wl.total_q, wl.num_heads, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((wl.total_q, wl.num_heads), dtype=torch.float32, device=dev)
        self.ws = torch.empty(mtv.workspace_bytes(wl.bs, mq, wl.num_heads), dtype=torch.uint8,
                              device=dev)
        d = self.d
        self.args_call = (d["q"], d["kv_cache"], d["kv_indices"], d["kv_indptr"],
                          d["out_cache_loc"], d["custom_mask"], d["mask_indptr"],
                          d["qo_indptr"], wl.sm_scale, self.out, self.lse, self.ws, mq)

    def call(self, stream=None):
        if self.lanes:   # a lane count other than the library's: the debug entry point
            self.mtv.mla_tree_verify_debug_ex(*self.args_call, lanes=self.lanes, stream=stream)
        else:
            self.mtv.mla_tree_verify(*self.args_call, stream=stream)

    def profiled(self, ev, stream):
        if self.lanes:   # no per-kernel events on this path: the whole call as "split"
            ev[0].record(stream)
            ev[1].record(stream)
            self.call(stream)
            ev[2].record(stream)
        else:
            self.mtv.binding.mla_tree_verify_profiled(*self.args_call, ev, stream=stream)

    def status(self):
        return self.mtv.read_device_status(self.ws)


def graph_steps(stream, flush, n_steps, n_events, body):
    """CUDA graphs of up to 50 steps each: an L2 flush (256 MiB write, outside the events),
    then body(events) of one step.  Events recorded inside a capture are external ones so
    that they can be read after a replay.  The graphs are replayed once before return."""
    import torch
    graphs, left = [], n_steps
    while left > 0:
        n = min(50, left)
        ev = [[_timing_event() for _ in range(n_events)] for _ in range(n)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for row in ev:       # torch creates the CUDA event on its first record
                for e in row:
                    e.record()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    flush.zero_()
                    body(ev[i])
        graphs.append((g, ev))
        left -= n
    for g, _ in graphs:
        g.replay()
    torch.cuda.synchronize()
    return graphs


def replay_times(graphs, pairs):
    """Replays the graphs; per step, the elapsed ms between each (i, j) event pair."""
    import torch
    out = [[] for _ in pairs]
    for g, ev in graphs:
        g.replay()
        torch.cuda.synchronize()
        for e in ev:
            for k, (i, j) in enumerate(pairs):
                out[k].append(e[i].elapsed_time(e[j]))
    return out


def per_kernel_times(vs, stream, flush, steps):
    """Planner and split-kernel time of a call from events between the two kernels (a
    separate replay: the event between them keeps them from overlapping)."""
    import statistics
    graphs = graph_steps(stream, flush, steps, 3, lambda ev: vs.profiled(ev, stream))
    plan, split = replay_times(graphs, [(0, 1), (1, 2)])
    return statistics.mean(plan), statistics.mean(split)


def roofline_of(c, split_ms, t_call_s):
    """The split kernel's binding roofline (tensor: flops / bf16 peak; HBM: KV bytes read
    once / copy peak, whichever takes longer at peak), and the call's."""
    hbm_gbs, tc_tflops, src = peaks()
    tensor_bound = c["flops"] / (tc_tflops * 1e12) >= c["kv_bytes"] / (hbm_gbs * 1e9)
    if tensor_bound:
        roof = {"bound": "tensor", "kernel": "split",
                "achieved": c["flops"] / (split_ms * 1e-3) / 1e12, "peak": tc_tflops,
                "unit": "TFLOP/s", "peak_source": f"{src} bf16 dense (burst)"}
    else:
        roof = {"bound": "hbm", "kernel": "split",
                "achieved": c["kv_bytes"] / (split_ms * 1e-3) / 1e9, "peak": hbm_gbs,
                "unit": "GB/s", "peak_source": f"{src} HBM copy (burst)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    call = {"t_hbm_us": c["kv_bytes"] / (hbm_gbs * 1e9) * 1e6,
            "t_tensor_us": c["flops"] / (tc_tflops * 1e12) * 1e6,
            "frac_of_binding": max(c["kv_bytes"] / (hbm_gbs * 1e9),
                                   c["flops"] / (tc_tflops * 1e12)) / t_call_s,
            "peaks": src}
    return roof, call


def parity_sample(vs, n_rows, seed):
    """The oracle on a sample of (row, head) pairs against the call's last outputs:
    the largest |out - ref| / (1 + |ref|) and |lse - ref|."""
    import numpy as np
    import oracle
    wl = vs.wl
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, wl.total_q, n_rows), rng.integers(0, wl.num_heads, n_rows)], 1)
    ref_out, ref_lse = oracle.Oracle(wl).attend(rows, threads=os.cpu_count() or 1)
    r, h = rows[:, 0], rows[:, 1]
    got = vs.out.float().cpu().numpy()[r, h].astype(np.float64)
    got_lse = vs.lse.cpu().numpy()[r, h].astype(np.float64)
    e_out = float((np.abs(got - ref_out) / (1 + np.abs(ref_out))).max())
    fin = np.isfinite(ref_lse)
    e_lse = float(np.abs(got_lse[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    return {"pairs": int(n_rows), "max_out_err": e_out, "max_lse_err": e_lse,
            "within_tolerance": bool(e_out <= 1e-2 and e_lse <= 1e-3)}


def measure_config(k, args, dev, stream, flush):
    """One of the five verify configs at 1 GPU: µs per call (CUDA-graph replays, L2
    flushed between calls), KV GB/s, TFLOP/s, the binding-roofline fractions, a sampled
    parity check and the fp64 oracle timed on the host cores."""
    import statistics
    import torch
    from mla_tree_verify_gb300 import workloads as W
    wl = W.shape(k)
    vs = VerifySetup(wl, dev)
    for _ in range(args.warmup):
        flush.zero_()
        vs.call()
    torch.cuda.synchronize()
    status = vs.status()
    steps = 100   # at most 0.6 ms a call on configs 1-4: 100 replays cost well under a second
    graphs = graph_steps(stream, flush, steps, 2, lambda ev: (
        ev[0].record(stream), vs.call(stream), ev[1].record(stream)))
    (tot,) = replay_times(graphs, [(0, 1)])
    plan_ms, split_ms = per_kernel_times(vs, stream, flush, 20)
    us = statistics.mean(tot) * 1e3
    c = workload_counts(wl)
    roof, call = roofline_of(c, split_ms, us * 1e-6)
    entry = {"workload": W.SHAPE_NAMES[k], "us_per_call": us,
             "us_per_call_median": statistics.median(tot) * 1e3, "split_us": split_ms * 1e3,
             "plan_us": plan_ms * 1e3, "kv_gbs": c["kv_bytes"] / (us * 1e-6) / 1e9,
             "tflops": c["flops"] / (us * 1e-6) / 1e12, "bound": roof["bound"],
             "frac_of_binding_call": call["frac_of_binding"],
             "split_kernel_frac": roof["frac"], "steps": steps, "device_status": status,
             "parity_sample": parity_sample(vs, 64, seed=k)}
    if not args.no_cpu_baseline:
        entry["oracle"] = cpu_baseline(wl, args.per_config_cpu_seconds)
    del vs, graphs
    torch.cuda.empty_cache()
    return entry



def bench_verify(args, wl, name):
    """The verify call on one workload (by default the largest single-GPU config) as
    CUDA-graph replays with L2 flushed between calls; N replicas under torchrun.  Rank 0
    prints one JSON line, with the five configs measured one after another under
    `per_config` (1 GPU, rank 0 only)."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import mla_tree_verify_gb300 as mtv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    mtv.prepare()
    vs = VerifySetup(wl, dev, lanes=args.lanes)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.zero_()
        vs.call()
    torch.cuda.synchronize()
    if vs.status() != 0:
        raise RuntimeError("device error flags set")

    K = args.steps
    # The timed steps run as CUDA-graph replays (the call is capture-safe; this is how a
    # serving loop replays it): per step an L2 flush outside the events, then the call
    # between two events.
    stream = torch.cuda.Stream()
    _timing_event()                  # settles _EXTERNAL_EVENTS
    if _EXTERNAL_EVENTS:
        graphs = graph_steps(stream, flush, K, 2, lambda ev: (
            ev[0].record(stream), vs.call(stream), ev[1].record(stream)))
    else:                            # older torch: the call's own external events
        graphs = graph_steps(stream, flush, K, 3, lambda ev: vs.profiled(ev, stream))
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    (tot,) = replay_times(graphs, [(0, -1)])
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    if vs.status() != 0:
        raise RuntimeError("device error flags set")
    plan_ms, split_ms = per_kernel_times(vs, stream, flush, min(K, 20))
    t_sum = max_over_ranks(sum(tot), device=dev)
    # the floor of any two-kernel call: a CUDA graph of two empty kernels, replayed the
    # same way (the reference point for shapes far below a microsecond of work)
    floor = []
    fg = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(0)
        torch.cuda._sleep(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(fg, stream=stream):
            torch.cuda._sleep(0)
            torch.cuda._sleep(0)
    fg.replay()
    torch.cuda.synchronize()
    for _ in range(50):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fg.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        floor.append(e0.elapsed_time(e1))
    # the same call launched eagerly (context: launch gap between the two kernels)
    eager = []
    for _ in range(10):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        vs.call()
        e1.record()
        torch.cuda.synchronize()
        eager.append(e0.elapsed_time(e1))
    us_per_call = whole_job_us_per_call(t_sum, K, world)

    # end to end through the same C-ABI call with host buffers (pinned), copies timed
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory()
              for k, v in vs.host.items()}
    out_h = torch.empty(vs.out.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty(vs.lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    e2e = []
    for i in range(args.e2e_steps + 3):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in vs.d:
            vs.d[k].view(torch.uint8).copy_(pinned[k].view(torch.uint8), non_blocking=True)
        vs.call()
        out_h.copy_(vs.out, non_blocking=True)
        lse_h.copy_(vs.lse, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            e2e.append(e0.elapsed_time(e1))
    e2e_us = statistics.mean(e2e) * 1e3
    del pinned

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    c = workload_counts(wl)
    t_call = us_per_call * world * 1e-6
    roof, roof_call = roofline_of(c, split_ms, t_call)
    roof["traffic"] = split_kernel_traffic(name, c["kv_bytes"])
    roof["algorithmic_flops_per_launch"] = c["flops"]
    roof["algorithmic_kv_bytes_per_launch"] = c["kv_bytes"]
    line = {
        "metric": METRIC, "value": us_per_call, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_sum / K, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl, name),
        "kv_gbs": c["kv_bytes"] / t_call / 1e9,
        "tflops": c["flops"] / t_call / 1e12,
        "roofline_call": roof_call,
        "kernels_us": {"plan": plan_ms * 1e3, "split": split_ms * 1e3},
        "timing": "CUDA-graph replay, events around the call; per-kernel times from a "
                  "separate replay with events between the kernels; eager launch for context",
        "median_us_per_call": statistics.median(tot) * 1e3,
        "eager_us_per_call": statistics.mean(eager) * 1e3,
        "floor_us_two_empty_kernels_graph": statistics.median(floor) * 1e3,
        "roofline": roof,
        "e2e": {"value": e2e_us, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * K,   # planner + split kernel per step (flush kernels not counted)
        "clocks": clk,
        "wall_s_timed_region": wall,
        "lanes": mtv.plan_header(vs.ws)["lanes"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if (not args.no_per_config and args.heads == 64 and args.layout == "scattered" and
            not args.lanes):
        from mla_tree_verify_gb300 import workloads as W
        head = {"workload": name, "us_per_call": us_per_call, "split_us": split_ms * 1e3,
                "plan_us": plan_ms * 1e3, "kv_gbs": line["kv_gbs"], "tflops": line["tflops"],
                "bound": roof["bound"], "frac_of_binding_call": roof_call["frac_of_binding"],
                "split_kernel_frac": roof["frac"], "steps": K, "device_status": vs.status(),
                "parity_sample": parity_sample(vs, 64, seed=args.shape)}
        if "cpu_baseline" in line:
            head["oracle"] = line["cpu_baseline"]
        del vs
        torch.cuda.empty_cache()
        per = {}
        for k in sorted(W.SHAPE_NAMES):
            per[str(k)] = head if k == args.shape else measure_config(k, args, dev, stream, flush)
        line["per_config"] = per
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--shape", type=int, default=5,
                    help="verify config 1..5 (5, the largest single-GPU one, is the headline)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--lanes", type=int, default=0, choices=[0, 1, 2, 4, 8],
                    help="CTAs per lane group of the work plan (0: the library's choice; "
                         "others run through the debug entry point, without per-kernel times)")
    ap.add_argument("--shape-bs", type=int, default=0,
                    help="a smaller draw of the shape's distribution with this many requests "
                         "(shapes 4 and 5; for profiling), instead of the shape itself")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config block (configs 1-5 measured one by one)")
    ap.add_argument("--per-config-cpu-seconds", type=float, default=3.0,
                    help="host seconds of oracle sampling per config in the per-config block")
    ap.add_argument("--heads", type=int, choices=[64, 8], default=64,
                    help="query heads per token: 64, or 8 (a tensor-parallel shard of 8 ranks)")
    ap.add_argument("--kernel", choices=["verify", "kv_gather", "conv1d"], default="verify",
                    help="kv_gather: the defragmentation copy of the shape's prefix rows; "
                         "conv1d: the conv-state update with a deduplicated window")
    ap.add_argument("--conv-bs", type=int, default=128, help="--kernel conv1d: requests")
    ap.add_argument("--conv-t", type=int, default=8, help="--kernel conv1d: draft tokens")
    ap.add_argument("--conv-types", default="bf16,bf16",
                    choices=["bf16,bf16", "bf16,f32", "f32,bf16", "f32,f32"],
                    help="--kernel conv1d: input and state element types")
    ap.add_argument("--conv-window", default="contiguous", choices=["contiguous", "transposed"],
                    help="--kernel conv1d: the window rows' layout ([slot][dim][T + 2], or "
                         "[T + 2][slot][dim] seen transposed)")
    ap.add_argument("--layout", choices=["scattered", "contiguous", "defrag"], default="scattered",
                    help="slots of the referenced rows: scattered over the pool (the bench), "
                         "consecutive (as after a defragmenting gather-copy), or scattered with "
                         "the gather-copy timed before every verify")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.kernel == "conv1d":
        (bench_conv1d if args.impl == "mine" else run_reference_conv1d)(args)
        return
    from mla_tree_verify_gb300 import workloads as W
    lay = "scattered" if args.layout == "defrag" else args.layout
    if args.shape_bs:
        wl = W.shape_sample(args.shape, args.shape_bs, heads=args.heads, layout=lay)
        name = wl.name
        args.no_per_config = True
    else:
        wl = W.shape(args.shape, heads=args.heads, layout=lay)
        name = W.SHAPE_NAMES[args.shape]
    name += ("" if args.heads == 64 else "_heads8") + ("" if args.layout == "scattered"
                                                      else "_" + args.layout)
    if args.impl == "reference":
        run_reference(args, wl, name)
        return
    if args.kernel == "kv_gather":
        bench_kv_gather(args, wl, name)
        return
    if args.layout == "defrag":
        bench_defrag_verify(args, wl, W.SHAPE_NAMES[args.shape])
        return
    bench_verify(args, wl, name)


if __name__ == "__main__":
    main()
