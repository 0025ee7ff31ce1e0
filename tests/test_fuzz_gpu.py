"""Randomised GPU sweeps: many small seeded workloads, every output checked against the
oracles.

Verify attention: random batch sizes, prefix and draft lengths (including empty prefixes
and single drafts), chain or random trees, scattered / contiguous / run slot layouts,
64 or 8 heads; and long prefixes whose split-heavy tokens merge in two levels.  Conv-state update: random batch sizes, T, dims, state lengths, accept
offsets, padded rows, bias and activation; then element types (bf16, fp32, mixed), any
channel count and strided views of the state and window.  The seeds are fixed, so a
failure reproduces.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle  # noqa: E402
import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import conv_workloads as CW  # noqa: E402
from mla_tree_verify_gb300 import workloads as W  # noqa: E402
from gpu_util import all_rows, check_rows, run, to_device  # noqa: E402
import test_conv1d_gpu as conv  # noqa: E402


@pytest.mark.parametrize("seed", range(48))
def test_verify_random_workloads(seed):
    rng = np.random.default_rng(7000 + seed)
    bs = int(rng.integers(1, 7))
    P = rng.integers(0, 700, size=bs)
    P[rng.random(bs) < 0.2] = 0
    T = rng.integers(1, 17, size=bs)
    tree = "chain" if rng.random() < 0.4 else "random"
    layout = ["scattered", "contiguous", "runs"][int(rng.integers(0, 3))]
    heads = 8 if rng.random() < 0.3 else 64
    pool = int(3 * (P.sum() + T.sum()) + 512)
    wl = W.build("fuzz", 7000 + seed, P, T, tree, pool, heads=heads, layout=layout)
    out, lse, ws = run(wl)
    assert mtv.read_device_status(ws) == 0
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))


@pytest.mark.parametrize("seed", range(16))
def test_verify_random_long_prefixes(seed):
    """Prefixes up to 40k keys with few draft tokens, so that many column groups are cut
    into more than 16 pieces and merge in two levels, next to short ones; every output
    against the oracle, and a second call must give the same bits."""
    rng = np.random.default_rng(9000 + seed)
    bs = int(rng.integers(1, 4))
    P = rng.integers(0, 40000, size=bs)
    P[rng.random(bs) < 0.2] = int(rng.integers(0, 300))
    heads = 8 if rng.random() < 0.4 else 64
    T = rng.integers(1, 20 if heads == 8 else 5, size=bs)
    tree = "chain" if rng.random() < 0.5 else "random"
    layout = ["scattered", "contiguous", "runs"][int(rng.integers(0, 3))]
    pool = int(3 * (P.sum() + T.sum()) + 512)
    wl = W.build("fuzzlong", 9000 + seed, P, T, tree, pool, heads=heads, layout=layout)
    d = to_device(wl)
    out, lse, ws = run(wl, d)
    assert mtv.read_device_status(ws) == 0
    out2, lse2, _ = run(wl, d)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    ref_out, ref_lse = oracle.Oracle(wl).attend()
    check_rows(out, lse, ref_out, ref_lse, all_rows(wl))


@pytest.mark.parametrize("seed", range(48))
def test_conv_random_cases(seed):
    rng = np.random.default_rng(8000 + seed)
    bs = int(rng.integers(1, 40))
    T = int(rng.integers(1, 17))
    dim = 8 * int(rng.integers(1, 300))
    state_len = int(rng.choice([3, 3, 4, 7, 32]))
    c = CW.case(8000 + seed, bs=bs, T=T, dim=dim, state_len=state_len,
                accept=bool(rng.random() < 0.5), pad_rows=int(rng.integers(0, 3)),
                bias=bool(rng.random() < 0.7), silu=bool(rng.random() < 0.7),
                num_slots=bs + int(rng.integers(0, 20)))
    conv.check(c, conv.run(c))


@pytest.mark.parametrize("seed", range(32))
def test_conv_general_random_cases(seed):
    """Random element types, channel counts (any, not only multiples of 8) and views."""
    import test_conv1d_general_gpu as gen
    rng = np.random.default_rng(8500 + seed)
    bs = int(rng.integers(1, 30))
    T = int(rng.integers(1, 17))
    dim = int(rng.integers(1, 1500))
    state_len = int(rng.choice([3, 4, 9, 32]))
    xd, sd = gen.TYPES[int(rng.integers(0, 4))]
    c = CW.case(8500 + seed, bs=bs, T=T, dim=dim, state_len=state_len,
                accept=bool(rng.random() < 0.5), pad_rows=int(rng.integers(0, 3)),
                bias=bool(rng.random() < 0.7), silu=bool(rng.random() < 0.7),
                num_slots=bs + int(rng.integers(0, 20)), x_dtype=xd, state_dtype=sd)
    wl = ["contiguous", "transposed", "padded_cols", "padded_slots"][int(rng.integers(0, 4))]
    sl = "channel_last" if rng.random() < 0.3 else "contiguous"
    gen.check(c, gen.run(c, wl, sl))
