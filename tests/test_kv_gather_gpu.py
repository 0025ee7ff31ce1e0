"""GPU tests of the KV gather-copy (the defragmentation step), through the C ABI.

The CUDA gather must match the oracle's gather bit for bit (rows, new indices, the count
of out-of-pool slots); a verify call that reads the gathered rows through the new
indices must return exactly what it returns on the scattered layout.
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
from gpu_util import run, to_device  # noqa: E402


def _pool(rng, slots):
    bits = rng.standard_normal((slots, 576)).astype(np.float32).view(np.uint32) >> 16
    return bits.astype(np.uint16)


def _gather(kv, idx, ptr, dst_rows, dst_slot0, num_slots=None, fill=0x7FC0):
    d_kv = torch.from_numpy(kv.view(np.int16)).cuda().view(torch.bfloat16)
    d_idx = torch.from_numpy(np.asarray(idx, dtype=np.int32)).cuda()
    d_ptr = torch.from_numpy(np.asarray(ptr, dtype=np.int32)).cuda()
    dst = torch.full((dst_rows, 576), fill, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    new = torch.full_like(d_idx, -7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mtv.kv_gather(d_kv, d_idx, d_ptr, dst, dst_slot0, new, status, num_slots=num_slots)
    torch.cuda.synchronize()
    return (dst.view(torch.int16).cpu().numpy().view(np.uint16), new.cpu().numpy(),
            int(status.item()))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_matches_the_oracle_bit_for_bit(seed):
    rng = np.random.default_rng(seed)
    slots = 5000
    kv = _pool(rng, slots)
    n = int(rng.integers(1, 4000))
    idx = rng.permutation(slots)[:n].astype(np.int32)
    cuts = np.sort(rng.integers(0, n + 1, size=int(rng.integers(1, 12))))
    ptr = np.concatenate([[0], cuts, [n]]).astype(np.int32)       # some requests empty
    dst, new, st = _gather(kv, idx, ptr, n + 5, 123)
    ref, ref_new, bad = oracle.kv_gather(kv, idx, ptr, n + 5, 123)
    assert st == 0 and bad == 0
    assert np.array_equal(dst[:n], ref[:n])
    assert (dst[n:] == 0x7FC0).all()                             # rows past the batch untouched
    assert np.array_equal(new, ref_new)


def test_batch_offset_and_ragged_rows():
    # kv_indptr[0] > 0, a row count that is not a multiple of the 4-row step
    rng = np.random.default_rng(9)
    kv = _pool(rng, 300)
    idx = rng.integers(0, 300, size=57).astype(np.int32)
    ptr = np.array([6, 6, 13, 50], dtype=np.int32)
    dst, new, st = _gather(kv, idx, ptr, 44, 7)
    ref, ref_new, _ = oracle.kv_gather(kv, idx, ptr, 44, 7)
    assert st == 0
    assert np.array_equal(dst, ref)
    assert np.array_equal(new[6:50], ref_new[6:50])
    assert (new[:6] == -7).all() and (new[50:] == -7).all()      # outside the batch: untouched


def test_out_of_pool_slots_give_zero_rows_and_a_flag():
    rng = np.random.default_rng(4)
    kv = _pool(rng, 100)
    idx = np.array([5, 100, 7, -2, 99, 3], dtype=np.int32)
    dst, new, st = _gather(kv, idx, [0, 6], 6, 0)
    ref, ref_new, bad = oracle.kv_gather(kv, idx, [0, 6], 6, 0)
    assert bad == 2 and st == mtv.GATHER_BAD_SLOT
    assert np.array_equal(dst, ref) and np.array_equal(new, ref_new)


def test_bad_extent_copies_nothing():
    rng = np.random.default_rng(5)
    kv = _pool(rng, 100)
    idx = np.arange(20, dtype=np.int32)
    # too few destination rows, decreasing, negative, and past the end of kv_indices
    for ptr, rows in (([0, 20], 19), ([5, 2], 30), ([-1, 4], 30), ([0, 25], 30)):
        dst, new, st = _gather(kv, idx, ptr, rows, 0)
        assert st == mtv.GATHER_BAD_ARGS
        assert (dst == 0x7FC0).all() and (new == -7).all()


def test_graph_replay_with_new_indices():
    rng = np.random.default_rng(6)
    slots, n = 4000, 1500
    kv = _pool(rng, slots)
    d_kv = torch.from_numpy(kv.view(np.int16)).cuda().view(torch.bfloat16)
    d_idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    d_ptr = torch.tensor([0, 600, 1500], dtype=torch.int32, device="cuda")
    dst = torch.zeros((n, 576), dtype=torch.bfloat16, device="cuda")
    new = torch.zeros(n, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mtv.prepare()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        mtv.kv_gather(d_kv, d_idx, d_ptr, dst, 0, new, status, stream=s)   # warm-up
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            mtv.kv_gather(d_kv, d_idx, d_ptr, dst, 50, new, status, stream=s)
    for seed in (10, 11):
        idx = np.random.default_rng(seed).permutation(slots)[:n].astype(np.int32)
        d_idx.copy_(torch.from_numpy(idx))
        g.replay()
        torch.cuda.synchronize()
        ref, ref_new, _ = oracle.kv_gather(kv, idx, [0, 600, 1500], n, 50)
        assert np.array_equal(dst.view(torch.int16).cpu().numpy().view(np.uint16), ref)
        assert np.array_equal(new.cpu().numpy(), ref_new)
    assert int(status.item()) == 0


@pytest.mark.parametrize("shape_id", [2, 4])
def test_verify_reads_the_gathered_rows_bit_identically(shape_id):
    """Gather a verify workload's prefix rows to the end of an enlarged pool; the verify
    call on (enlarged pool, new indices) must equal the call on the scattered layout."""
    wl = W.shape(shape_id)
    out1, lse1, _ = run(wl)
    d = to_device(wl)
    slots = d["kv_cache"].shape[0]
    n = d["kv_indices"].numel()
    pool = torch.empty((slots + n, 576), dtype=torch.bfloat16, device="cuda")
    pool[:slots].copy_(d["kv_cache"])
    new = torch.empty_like(d["kv_indices"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mtv.kv_gather(d["kv_cache"], d["kv_indices"], d["kv_indptr"], pool[slots:], slots, new, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # sampled entries against the definition
    sample = torch.randint(0, n, (256,), device="cuda")
    assert torch.equal(pool[slots + sample].view(torch.int16),
                       d["kv_cache"][d["kv_indices"][sample].long()].view(torch.int16))
    assert torch.equal(new, torch.arange(slots, slots + n, dtype=torch.int32, device="cuda"))
    d2 = dict(d)
    d2["kv_cache"] = pool
    d2["kv_indices"] = new
    out2, lse2, _ = run(wl, d2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_gather_then_verify_in_one_graph():
    """The gather-copy and the verify call on the rewritten indices, captured together in
    one CUDA graph and replayed with new prefix indices, match the oracle."""
    wl = W.build("gv", 31, [300, 129, 700], [16, 3, 9], "random", 4096)
    d = to_device(wl)
    slots = d["kv_cache"].shape[0]
    n = d["kv_indices"].numel()
    pool = torch.empty((slots + n, 576), dtype=torch.bfloat16, device="cuda")
    pool[:slots].copy_(d["kv_cache"])
    new = torch.empty_like(d["kv_indices"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    from gpu_util import alloc_outputs, check_rows, all_rows
    out, lse, ws, mq = alloc_outputs(wl)

    def step(stream):
        mtv.kv_gather(pool, d["kv_indices"], d["kv_indptr"], pool[slots:], slots, new, status,
                      num_slots=slots, stream=stream)
        mtv.mla_tree_verify(d["q"], pool, new, d["kv_indptr"], d["out_cache_loc"],
                            d["custom_mask"], d["mask_indptr"], d["qo_indptr"], wl.sm_scale, out,
                            lse, ws, mq, stream=stream)
    mtv.prepare()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step(s)
    # new prefix slots: a permutation of the prefix rows inside the original pool
    rng = np.random.default_rng(32)
    perm = rng.permutation(n)
    wl2 = W.build("gv", 31, [300, 129, 700], [16, 3, 9], "random", 4096)
    wl2.kv_indices = np.ascontiguousarray(wl.kv_indices[perm])
    d["kv_indices"].copy_(torch.from_numpy(wl2.kv_indices))
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and mtv.read_device_status(ws) == 0
    ref_out, ref_lse = oracle.Oracle(wl2).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl2))
