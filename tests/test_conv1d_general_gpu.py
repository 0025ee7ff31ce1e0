"""GPU parity of the general conv-state update: fp32 and bf16 inputs and state in any mix,
any channel count, strided views of the conv state and of the window rows
(causal_conv1d_update_dedup_ex).

The pull request "jianc99/sglang#1", section "Accuracy Tests", covers fp32 and bf16, mixed
input and state dtypes, transposed window views and a channel count that leaves a partial
channel block; these tests cover the same against the fp64 oracle.  Window rows and state
must match bit for bit (they are the row's values stored in the state type); outputs must
lie within the bound of their type:
  * bf16 out: one bf16 ulp of the exact value (2^-8 |ref|), plus 1e-5;
  * fp32 out: 2^-18 (|ref| + |bias| + sum_k |w_k f_k|): the fp32 multiply-adds err by a few
    units of 2^-24 of the summed magnitudes, and the fast exponential and divide of the SiLU
    by a few units of 2^-21 of the result.
Entries of the buffers outside the views, rows of padded requests and slots that no
request names must stay untouched.
"""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle.conv1d as O  # noqa: E402
import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import conv_workloads as CW  # noqa: E402

TYPES = [("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16"), ("f32", "f32")]


def to_dev(a):
    """numpy (bf16 bits as uint16, fp32, int32) -> CUDA tensor of the same values."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def bits(t):
    """A tensor's element bits as numpy (uint16 for bf16, uint32 for fp32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def np_bits(a):
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


def fill_bits(dtype):
    return CW.SENTINEL if dtype == torch.bfloat16 else CW.SENTINEL_F32


def make_view(logical, layout, T):
    """A device view with the logical contents and the given physical layout; returns
    (view, physical buffer, mask of the physical entries outside the view)."""
    n, dim, cols = logical.shape
    dt = torch.bfloat16 if logical.dtype == np.uint16 else torch.float32
    if layout == "contiguous":
        phys = to_dev(logical)
        return phys, phys, None
    if layout == "transposed":                   # columns outermost: [cols][slots][dim]
        phys = torch.empty((cols, n, dim), dtype=dt, device="cuda")
        view = phys.permute(1, 2, 0)
    elif layout == "padded_cols":                # each row padded by 3 entries
        phys = torch.empty((n, dim, cols + 3), dtype=dt, device="cuda")
        view = phys[:, :, :cols]
    elif layout == "padded_slots":               # each slot's block followed by 40 entries
        phys = torch.empty((n, dim * cols + 40), dtype=dt, device="cuda")
        view = phys[:, :dim * cols].view(n, dim, cols)
    else:
        raise ValueError(layout)
    ib = torch.int16 if dt == torch.bfloat16 else torch.int32
    sentinel = int(np.array(fill_bits(dt)).astype(np.int64))
    sentinel = sentinel - (1 << 16) if (dt == torch.bfloat16 and sentinel >= 1 << 15) else sentinel
    phys.view(ib).fill_(sentinel)
    view.copy_(to_dev(logical))
    outside = torch.ones(phys.shape, dtype=torch.bool, device="cuda")
    if layout == "transposed":
        outside.zero_()
    elif layout == "padded_cols":
        outside[:, :, :cols] = False
    else:
        outside[:, :dim * cols] = False
    return view, phys, outside


def run(c, window_layout="contiguous", state_layout="contiguous", stream=None):
    d = dict(x=to_dev(c.x), w=to_dev(c.weight), b=to_dev(c.bias), slots=to_dev(c.slots),
             acc=to_dev(c.num_accept), out=to_dev(c.out),
             status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    d["win"], d["win_phys"], d["win_out"] = make_view(c.window, window_layout, c.T)
    if state_layout == "channel_last":   # [slots][state_len][dim] seen as [slots][dim][state_len]
        phys = to_dev(np.ascontiguousarray(np.transpose(c.conv_state, (0, 2, 1))))
        d["st"] = phys.permute(0, 2, 1)
    else:
        d["st"] = to_dev(c.conv_state)
    mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                      d["status"], silu=c.silu, stream=stream)
    torch.cuda.synchronize()
    return d


def _magnitude(c, b):
    """|bias| + sum_k |w_k f_k| per output of request b, [T, dim]."""
    slot = int(c.slots[b])
    o = 0 if c.num_accept is None else int(c.num_accept[b]) - 1
    f = np.concatenate([O.as_f64(c.conv_state[slot][:, o:o + 3]), O.as_f64(c.x[b]).T], axis=1)
    bias = None if c.bias is None else np.abs(O.as_f64(c.bias))
    return O.conv_outputs(np.abs(f), np.abs(O.as_f64(c.weight)), bias, False)


def check(c, d):
    ref_out, ref_state, ref_win = O.update(c)
    assert int(d["status"].item()) == 0
    np.testing.assert_array_equal(bits(d["win"]), np_bits(ref_win))
    np.testing.assert_array_equal(bits(d["st"]), np_bits(ref_state))
    if d["win_out"] is not None:
        outside = bits(d["win_phys"])[d["win_out"].cpu().numpy()]
        assert (outside == fill_bits(d["win"].dtype)).all()
    got = bits(d["out"])
    for b in range(c.bs):
        if c.slots[b] == CW.PAD_SLOT:
            assert (got[b] == np_bits(np.asarray(c.out[b]))).all()
            continue
        r = ref_out[b]
        if c.x_dtype == "bf16":
            g = O.bf16_to_f64(got[b])
            bound = np.ldexp(np.abs(r), -8) + 1e-5
        else:
            g = got[b].view(np.float32).astype(np.float64)
            bound = np.ldexp(np.abs(r) + _magnitude(c, b), -18)
        err = np.abs(g - r)
        assert (err <= bound).all(), f"request {b}: max err {err.max():.3e}"


@pytest.mark.parametrize("xd,sd", TYPES)
@pytest.mark.parametrize("T,dim,bs,state_len", [(1, 13, 3, 3), (3, 129, 5, 7), (8, 1000, 4, 4),
                                                 (9, 260, 3, 32), (16, 385, 2, 5)])
def test_types_and_partial_channel_blocks(xd, sd, T, dim, bs, state_len):
    c = CW.case(900 + T + dim, bs=bs, T=T, dim=dim, state_len=state_len,
                accept=state_len > 3, pad_rows=1 if bs > 2 else 0, x_dtype=xd, state_dtype=sd)
    check(c, run(c))


@pytest.mark.parametrize("xd,sd", TYPES)
@pytest.mark.parametrize("window_layout,state_layout", [
    ("transposed", "contiguous"), ("padded_cols", "contiguous"), ("padded_slots", "contiguous"),
    ("contiguous", "channel_last"), ("transposed", "channel_last")])
def test_strided_views(xd, sd, window_layout, state_layout):
    c = CW.case(950, bs=6, T=5, dim=200, state_len=6, accept=True, pad_rows=1, x_dtype=xd,
                state_dtype=sd)
    check(c, run(c, window_layout, state_layout))


@pytest.mark.parametrize("T", [1, 2, 8, 16])
def test_general_path_equals_fast_path_bitwise(T):
    """bf16 everywhere with a multiple of 8 channels: contiguous rows and a transposed window
    (channel-contiguous columns) take the 4-channels-a-thread kernel, padded rows the general
    one; outputs, state and window rows agree bit for bit."""
    c = CW.case(960 + T, bs=7, T=T, dim=1024, state_len=5, accept=True, pad_rows=2)
    fast = run(c)
    for layout in ("transposed", "padded_cols"):
        other = run(c, layout)
        for key in ("out", "st", "win"):
            np.testing.assert_array_equal(bits(fast[key]), bits(other[key]),
                                          err_msg=f"{layout} {key}")
        check(c, other)


@pytest.mark.parametrize("T,dim", [(3, 8), (8, 1000), (16, 264)])
def test_transposed_window_bf16_state_len_3(T, dim):
    """The transposed window with bf16 state of length 3 (the bf16 kernel's state blocks
    are staged and stored whole), padded rows and a partial last warp."""
    c = CW.case(965 + T, bs=9, T=T, dim=dim, pad_rows=2)
    check(c, run(c, "transposed"))


@pytest.mark.parametrize("xd,dim", [("f32", 77), ("bf16", 80)])
def test_bad_slot_and_accept_general(xd, dim):
    """Status bits with a transposed window, on the general kernel (fp32 inputs) and on the
    bf16 kernel's column-major mode (bf16, 80 channels)."""
    c = CW.case(970, bs=4, T=4, dim=dim, state_len=5, accept=True, num_slots=10, x_dtype=xd)
    c.slots[1] = 10
    c.num_accept[2] = 4
    d = run(c, "transposed")
    assert int(d["status"].item()) == mtv.CONV1D_BAD_SLOT | mtv.CONV1D_BAD_ACCEPT
    got = bits(d["out"])
    for b in (1, 2):
        assert (got[b] == np_bits(np.asarray(c.out[b]))).all()
    ok = dataclasses.replace(c, slots=c.slots.copy())
    ok.slots[1] = CW.PAD_SLOT
    ok.slots[2] = CW.PAD_SLOT
    _, ref_state, ref_win = O.update(ok)
    np.testing.assert_array_equal(bits(d["st"]), np_bits(ref_state))
    np.testing.assert_array_equal(bits(d["win"]), np_bits(ref_win))


@pytest.mark.parametrize("xd,dim", [("f32", 301), ("bf16", 304)])
def test_graph_replay_general(xd, dim):
    """Graph replay with new inputs through a transposed window: the general kernel (fp32
    inputs) and the bf16 kernel's column-major mode (bf16, 304 channels)."""
    c = CW.case(980, bs=8, T=6, dim=dim, pad_rows=2, x_dtype=xd, state_dtype="bf16")
    d = run(c, "transposed")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    args = lambda: (d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                    d["status"])
    with torch.cuda.stream(s):
        mtv.conv1d_update(*args(), silu=c.silu, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            mtv.conv1d_update(*args(), silu=c.silu, stream=s)
    for seed in (981, 982):
        n = CW.case(seed, bs=8, T=6, dim=dim, pad_rows=2, num_slots=c.num_slots, x_dtype=xd,
                    state_dtype="bf16")
        n = dataclasses.replace(n, weight=c.weight, bias=c.bias)
        for key, arr in (("x", n.x), ("st", n.conv_state), ("slots", n.slots), ("win", n.window),
                         ("out", n.out)):
            d[key].copy_(to_dev(arr))
        d["status"].zero_()
        g.replay()
        torch.cuda.synchronize()
        check(n, d)


@pytest.mark.parametrize("xd", ["bf16", "f32"])
def test_largest_batch(xd):
    """65535 requests, the most one call takes (one grid row each): the bf16 case runs on
    the 4-channels-a-thread kernel, the fp32 one on the general kernel."""
    c = CW.case(990, bs=65535, T=2, dim=8, pad_rows=100, x_dtype=xd, state_dtype=xd)
    check(c, run(c))


def test_window_offsets_beyond_int32():
    """Window rows 2^29 + 64 elements apart, so that the last slots' rows start past 2^31
    elements (8.6 GB of bf16): the kernel's addresses must be 64-bit."""
    c = CW.case(991, bs=5, T=4, dim=64, num_slots=8, accept=True, state_len=4, pad_rows=1)
    stride = (1 << 29) + 64
    assert (c.num_slots - 1) * stride > 1 << 31
    phys = torch.empty((c.num_slots, stride), dtype=torch.bfloat16, device="cuda")
    win = phys[:, :c.dim * (c.T + 2)].view(c.num_slots, c.dim, c.T + 2)
    win.copy_(to_dev(c.window))
    d = dict(x=to_dev(c.x), w=to_dev(c.weight), b=to_dev(c.bias), slots=to_dev(c.slots),
             acc=to_dev(c.num_accept), out=to_dev(c.out), st=to_dev(c.conv_state), win=win,
             status=torch.zeros(1, dtype=torch.int32, device="cuda"), win_out=None)
    mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                      d["status"], silu=c.silu)
    torch.cuda.synchronize()
    check(c, d)
    del phys, win, d
    torch.cuda.empty_cache()


def test_transposed_window_offsets_beyond_int32():
    """A transposed window whose columns lie 2^29 elements apart (6.4 GB of bf16), so that
    columns 4 and 5 start past 2^31 elements; bf16 with channel-contiguous columns runs on
    the 4-channels-a-thread kernel."""
    c = CW.case(992, bs=5, T=4, dim=64, num_slots=8, pad_rows=1)
    col_stride = 1 << 29
    assert (c.T + 1) * col_stride > 1 << 31
    phys = torch.empty((c.T + 2, col_stride), dtype=torch.bfloat16, device="cuda")
    win = phys[:, :c.num_slots * c.dim].view(c.T + 2, c.num_slots, c.dim).permute(1, 2, 0)
    win.copy_(to_dev(c.window))
    d = dict(x=to_dev(c.x), w=to_dev(c.weight), b=to_dev(c.bias), slots=to_dev(c.slots),
             acc=to_dev(c.num_accept), out=to_dev(c.out), st=to_dev(c.conv_state), win=win,
             status=torch.zeros(1, dtype=torch.int32, device="cuda"), win_out=None)
    mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                      d["status"], silu=c.silu)
    torch.cuda.synchronize()
    check(c, d)
    del phys, win, d
    torch.cuda.empty_cache()
