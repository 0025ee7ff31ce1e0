"""GPU parity of the conv-state update with a deduplicated window (chain verify, K = 4).

Through the C ABI (causal_conv1d_update_dedup), against the fp64 oracle on the same seeded
inputs: the window rows and the conv state must match bit for bit (they are copies), the
outputs within one bf16 rounding of the exact value (the kernel computes in fp32 and
rounds to bf16, nearest even); rows of padded requests and slots that no request names
must stay untouched.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

import oracle.conv1d as O  # noqa: E402
import mla_tree_verify_gb300 as mtv  # noqa: E402
from mla_tree_verify_gb300 import conv_workloads as CW  # noqa: E402


def _dev(a, dt=torch.int16):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else a.dtype))
    t = t.cuda()
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def run(c, stream=None):
    d = dict(x=_dev(c.x), st=_dev(c.conv_state), w=_dev(c.weight), b=_dev(c.bias),
             slots=_dev(c.slots), acc=_dev(c.num_accept), win=_dev(c.window), out=_dev(c.out),
             status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                      d["status"], silu=c.silu, stream=stream)
    torch.cuda.synchronize()
    return d


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check(c, d):
    ref_out, ref_state, ref_win = O.update(c)
    assert int(d["status"].item()) == 0
    np.testing.assert_array_equal(bits(d["win"]), ref_win)
    np.testing.assert_array_equal(bits(d["st"]), ref_state)
    got = bits(d["out"])
    for b in range(c.bs):
        if c.slots[b] == CW.PAD_SLOT:
            assert (got[b] == CW.SENTINEL).all()
            continue
        g = O.bf16_to_f64(got[b])
        r = ref_out[b]
        err = np.abs(g - r)
        bound = np.ldexp(np.abs(r), -8) + 1e-5       # one bf16 ulp of |ref| (and a floor)
        assert (err <= bound).all(), f"request {b}: max err {err.max():.3e}"


@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 16])
@pytest.mark.parametrize("dim,bs", [(8, 1), (1000, 5), (2056, 3)])
def test_matches_oracle(T, dim, bs):
    c = CW.case(100 + T + dim, bs=bs, T=T, dim=dim, pad_rows=1 if bs > 2 else 0)
    check(c, run(c))


@pytest.mark.parametrize("state_len,T", [(4, 8), (6, 3), (12, 16), (32, 1)])
def test_accept_offsets_and_long_states(state_len, T):
    c = CW.case(200 + state_len, bs=6, T=T, dim=520, state_len=state_len, accept=True, pad_rows=1)
    check(c, run(c))


@pytest.mark.parametrize("bias,silu", [(False, False), (True, False), (False, True)])
def test_bias_and_activation_variants(bias, silu):
    c = CW.case(300, bs=4, T=5, dim=264, bias=bias, silu=silu)
    check(c, run(c))


def test_bad_slot_and_accept_set_flags_and_store_nothing():
    c = CW.case(400, bs=4, T=4, dim=64, state_len=5, accept=True, num_slots=10)
    c.slots[1] = 10                    # out of range
    c.num_accept[2] = 4                # offset 3 > state_len - 3
    d = run(c)
    st = int(d["status"].item())
    assert st == mtv.CONV1D_BAD_SLOT | mtv.CONV1D_BAD_ACCEPT
    got = bits(d["out"])
    assert (got[1] == CW.SENTINEL).all() and (got[2] == CW.SENTINEL).all()
    # the other two requests are computed as usual
    ok = CW.case(400, bs=4, T=4, dim=64, state_len=5, accept=True, num_slots=10)
    ok.slots[1] = CW.PAD_SLOT
    ok.slots[2] = CW.PAD_SLOT
    ref_out, ref_state, ref_win = O.update(ok)
    np.testing.assert_array_equal(bits(d["win"]), ref_win)
    np.testing.assert_array_equal(bits(d["st"]), ref_state)


def test_graph_replay_with_new_inputs():
    c = CW.case(500, bs=8, T=8, dim=1024, pad_rows=2)
    d = run(c)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                          d["status"], silu=c.silu, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"],
                              d["out"], d["status"], silu=c.silu, stream=s)
    for seed in (501, 502):
        n = CW.case(seed, bs=8, T=8, dim=1024, pad_rows=2, num_slots=c.num_slots)
        for key, arr in (("x", n.x), ("st", n.conv_state), ("slots", n.slots), ("win", n.window),
                         ("out", n.out)):
            d[key].copy_(_dev(arr))
        n.weight, n.bias = c.weight, c.bias
        g.replay()
        torch.cuda.synchronize()
        check(n, d)


@pytest.mark.parametrize("bs,T", CW.BENCH_ROWS)
def test_bench_shapes(bs, T):
    c = CW.case(600 + bs + T, bs=bs, T=T, dim=CW.BENCH_DIM)
    check(c, run(c))


def test_consecutive_calls_chain_the_state():
    """Two calls on the same pool (the second reads the state the first wrote, in place)
    match the oracle applied twice; the second call's window rows replace the first's."""
    c1 = CW.case(700, bs=6, T=5, dim=264, pad_rows=1, state_len=4)
    d = run(c1)
    _, ref_state1, ref_win1 = O.update(c1)
    c2 = CW.case(701, bs=6, T=5, dim=264, pad_rows=1, state_len=4, num_slots=c1.num_slots)
    c2.slots, c2.weight, c2.bias = c1.slots, c1.weight, c1.bias
    c2.conv_state = ref_state1
    d["x"].copy_(_dev(c2.x))
    d["out"].copy_(_dev(c2.out))
    d["status"].zero_()
    mtv.conv1d_update(d["x"], d["st"], d["w"], d["b"], d["slots"], d["acc"], d["win"], d["out"],
                      d["status"], silu=c2.silu)
    torch.cuda.synchronize()
    c2.window = ref_win1                # the rows the first call left
    ref_out2, ref_state2, ref_win2 = O.update(c2)
    assert int(d["status"].item()) == 0
    np.testing.assert_array_equal(bits(d["st"]), ref_state2)
    np.testing.assert_array_equal(bits(d["win"]), ref_win2)
    got = bits(d["out"])
    for b in range(c2.bs):
        if c2.slots[b] == CW.PAD_SLOT:
            continue
        err = np.abs(O.bf16_to_f64(got[b]) - ref_out2[b])
        assert (err <= np.ldexp(np.abs(ref_out2[b]), -8) + 1e-5).all()
