"""Host-side check of the split kernel's work plan (no GPU).

The plan is restated here in Python from its rules:

- a column group is gt draft tokens (gt = 1 with 64 heads, 8 with 8 heads); request b
  has ncg = ceil(T_b / gt) of them and tiles = ceil(L_b / 128) key tiles;
- the split CTAs form lane groups of w consecutive CTAs; a job takes w column groups of
  one request, one per lane, over all of the request's tiles; the request's last job
  takes the nt column groups left and splits each one's tiles into k = w // nt
  sub-ranges of sl = ceil(tiles / k) tiles (lane r: column group r % nt, sub-range
  r // nt; lanes r >= nt k idle);
- a job occupies sl + SEG_COST units; units are numbered request by request, job by
  job; lane group g owns units [g C, (g + 1) C) with C = max(ceil(U / groups),
  ceil(max_tiles / (64 - 2 w)), min(max_tiles, 3) + SEG_COST, 1);
- each active lane of each job gets a lane-token index tok (request after request, job
  after job: cum_tok[b] + j w + r), and its piece in lane group g is written to partial
  slot tok + w g; a column group's pieces are its sub-ranges cut by lane groups, in that
  order, and its merge reads them through that numbering.

The test walks every lane's units as the kernel does and checks:

- every (column group, key tile) pair is computed exactly once, and empty units never;
- each column group's pieces are numbered 0 .. nseg - 1 in tile order, and sit in the
  slots its merge reads (piece i of the slot map);
- no two partials share a slot, and the slots stay below the workspace's slot count,
  bs * (ceil(max_q / gt) + 7) + grid;
- no column group is cut into more than 64 pieces;
- in a full job, the lanes of a group process the same key tiles at the same units (the
  draft tokens of a request read each tile together);
- with one lane per group the pieces are those of the token-by-token plan.
"""
import math
import random

import pytest

TILE = 128
NSPLIT = 64
SEG_COST = 1
MAX_LANES = 8


def geo(L, T, gt, w):
    ncg = -(-T // gt)
    tiles = -(-L // TILE)
    jobs = -(-ncg // w)
    nt_last = ncg - (jobs - 1) * w
    k_last = w // nt_last
    sl_last = -(-tiles // k_last)
    return dict(ncg=ncg, tiles=tiles, hf=tiles + SEG_COST, jobs=jobs, nt_last=nt_last,
                k_last=k_last, sl_last=sl_last)


def job_shape(g, j, w):
    if j == g["jobs"] - 1:
        return g["nt_last"], g["k_last"], g["sl_last"]
    return w, 1, g["tiles"]


def sub_len(tiles, s, sl):
    return max(0, min(sl, tiles - s * sl))


def plan(T, L, grid, w, gt=1):
    geos = [geo(l, t, gt, w) if t > 0 else None for t, l in zip(T, L)]
    cum = [0]
    for g in geos:
        units = 0 if g is None else (g["jobs"] - 1) * g["hf"] + g["sl_last"] + SEG_COST
        cum.append(cum[-1] + units)
    U = cum[-1]
    groups = grid // w
    maxt = max([g["tiles"] for g in geos if g is not None], default=0)
    C = max(-(-U // groups), -(-maxt // (NSPLIT - 2 * w)), min(maxt, 3) + SEG_COST, 1)
    cum_tok = [0]
    for g in geos:
        n = 0 if g is None else (g["jobs"] - 1) * w + g["nt_last"] * g["k_last"]
        cum_tok.append(cum_tok[-1] + n)
    return geos, cum, U, C, groups, cum_tok


def unit_request(cum, u):
    # the largest b with cum[b] <= u
    lo, hi = 0, len(cum) - 1
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if cum[mid] <= u:
            lo = mid
        else:
            hi = mid
    return lo


def seg_map(tok_b, j, w, cgl, js, tiles, nt, sl, C):
    """The slots of one column group's pieces, in order (sub-range, then lane group)."""
    ns = -(-tiles // sl)
    g_lo = js // C
    slots = []
    for s in range(ns):
        n = sub_len(tiles, s, sl)
        for g in range(g_lo, (js + n - 1) // C + 1):
            slots.append(tok_b + j * w + cgl + s * nt + w * g)
    return slots


def walk(T, L, grid, w, gt=1):
    """Every lane's segments: (group, lane, b, column group, tile0, tile1, first unit,
    slot, the column group's slots in order)."""
    geos, cum, U, C, groups, cum_tok = plan(T, L, grid, w, gt)
    segs = []
    for g in range(groups):
        for lane in range(w):
            u, u_end = g * C, min(U, (g + 1) * C)
            while u < u_end:
                b = unit_request(cum, u)
                ge = geos[b]
                j = min((u - cum[b]) // ge["hf"], ge["jobs"] - 1)
                js = cum[b] + j * ge["hf"]
                nt, k, sl = job_shape(ge, j, w)
                o0, o1 = u - js, min(u_end, js + sl + SEG_COST) - js
                assert o1 > o0
                u = js + o1
                if lane >= nt * k:
                    continue
                sub, cgl = lane // nt, lane % nt
                n = sub_len(ge["tiles"], sub, sl)
                if o0 >= n:
                    continue
                slots = seg_map(cum_tok[b], j, w, cgl, js, ge["tiles"], nt, sl, C)
                segs.append((g, lane, b, j * w + cgl, sub * sl + o0, sub * sl + min(o1, n),
                             js + o0, cum_tok[b] + j * w + lane + w * g, tuple(slots)))
    return segs, (geos, cum, U, C, groups, cum_tok)


def check(T, L, grid, w, gt=1, max_q=None):
    segs, (geos, cum, U, C, groups, cum_tok) = walk(T, L, grid, w, gt)
    assert C * groups >= U
    max_q = max_q or max(T + [1])
    slots_ws = len(T) * (-(-max_q // gt) + MAX_LANES - 1) + grid
    done = {}
    by_cg = {}
    for g, lane, b, cg, t0, t1, u0, slot, slots in segs:
        assert t1 > t0
        for t in range(t0, t1):
            key = (b, cg, t)
            assert key not in done, key
            done[key] = 1
        by_cg.setdefault((b, cg), []).append((t0, t1, slot, slots, g, lane, u0))
    for b, ge in enumerate(geos):
        if ge is None:
            continue
        for cg in range(ge["ncg"]):
            for t in range(ge["tiles"]):
                assert (b, cg, t) in done, (b, cg, t)
    used = set()
    for (b, cg), pieces in by_cg.items():
        pieces.sort()
        maps = {pc[3] for pc in pieces}
        assert len(maps) == 1
        slots = maps.pop()
        assert len(slots) == len(pieces) <= NSPLIT
        # pieces in tile order are the slot map's pieces 0 .. nseg - 1
        assert [pc[2] for pc in pieces] == list(slots)
        for pc in pieces:
            assert 0 <= pc[2] < slots_ws and pc[2] not in used
            used.add(pc[2])
    assert cum_tok[-1] + grid <= slots_ws
    # full jobs: every lane of a group processes the same tiles at the same units
    by_group_unit = {}
    for g, lane, b, cg, t0, t1, u0, slot, slots in segs:
        ge = geos[b]
        j = cg // w
        if j < ge["jobs"] - 1 or ge["nt_last"] == w:
            by_group_unit.setdefault((g, b, j), set()).add((t0, t1, u0))
    for key, ranges in by_group_unit.items():
        assert len(ranges) == 1, (key, ranges)
    return segs


def old_plan_pieces(T, L, grid):
    """The token-by-token plan: token t of request b has tiles + SEG_COST units; CTA k owns
    units [k C, (k + 1) C), C = max(ceil(U / grid), ceil(max_tiles / 63),
    min(max_tiles, 3) + SEG_COST, 1).  Returns {(b, t): [tile ranges]}."""
    tiles = [-(-l // TILE) if t > 0 else 0 for t, l in zip(T, L)]
    cum = [0]
    for t, n in zip(T, tiles):
        cum.append(cum[-1] + t * (n + SEG_COST))
    U = cum[-1]
    maxt = max([n for n, t in zip(tiles, T) if t > 0], default=0)
    C = max(-(-U // grid), -(-maxt // (NSPLIT - 1)), min(maxt, 3) + SEG_COST, 1)
    out = {}
    for b, t in enumerate(T):
        for i in range(t):
            u0 = cum[b] + i * (tiles[b] + SEG_COST)
            cuts = sorted({u0, u0 + tiles[b]} |
                          {k * C for k in range(grid + 1) if u0 < k * C < u0 + tiles[b]})
            out[(b, i)] = [(a - u0, c - u0) for a, c in zip(cuts, cuts[1:])]
    return out


@pytest.mark.parametrize("seed", range(60))
def test_random_plans(seed):
    rng = random.Random(seed)
    bs = rng.randint(1, 40)
    max_q = rng.randint(1, 24)
    T = [rng.randint(0, max_q) for _ in range(bs)]
    L = [rng.randint(1, 6000) + t for t in T]
    grid = rng.choice([8, 16, 40, 152])
    for w in (1, 2, 4, 8):
        check(T, L, grid, w, max_q=max_q)


@pytest.mark.parametrize("seed", range(10))
def test_random_plans_eight_heads(seed):
    rng = random.Random(100 + seed)
    bs = rng.randint(1, 20)
    max_q = rng.randint(1, 40)
    T = [rng.randint(0, max_q) for _ in range(bs)]
    L = [rng.randint(1, 3000) + t for t in T]
    for w in (1, 2, 4, 8):
        check(T, L, 152, w, gt=8, max_q=max_q)


@pytest.mark.parametrize("seed", range(20))
def test_one_lane_is_the_token_by_token_plan(seed):
    rng = random.Random(200 + seed)
    bs = rng.randint(1, 30)
    T = [rng.randint(0, 16) for _ in range(bs)]
    L = [rng.randint(1, 9000) + t for t in T]
    grid = rng.choice([7, 31, 152])
    segs = check(T, L, grid, 1)
    got = {}
    for g, lane, b, cg, t0, t1, *_ in segs:
        got.setdefault((b, cg), []).append((t0, t1))
    assert {k: sorted(v) for k, v in got.items()} == old_plan_pieces(T, L, grid)


def test_bench_like_shapes():
    rng = random.Random(7)
    for w in (1, 2, 4, 8):
        check([16] * 8, [rng.randint(1024, 4096) + 16 for _ in range(8)], 152, w)
        check([16], [185000 + 16], 152, w)
        check([8] * 32, [int(math.exp(rng.uniform(math.log(512), math.log(32768)))) + 8
                         for _ in range(32)], 152, w)
        T = [rng.choice([1, 4, 8, 16]) for _ in range(64)]
        check(T, [rng.randint(8192, 65536) + t for t in T], 152, w)
        check([4], [132], 152, w)


def test_small_batch_is_not_spread_one_tile_per_cta():
    # four drafts of two tiles each on 152 CTAs, one lane: C = 2 + SEG_COST, so every
    # token stays whole
    segs = check([4], [132], 152, 1)
    assert len(segs) == 4 and all(t1 - t0 == 2 for _, _, _, _, t0, t1, *_ in segs)
    # four lanes: the four drafts are one job, every lane has its whole token
    segs = check([4], [132], 152, 4)
    assert len(segs) == 4 and {s[1] for s in segs} == {0, 1, 2, 3}


def test_short_last_job_splits_tiles_among_idle_lanes():
    # 8 lanes, one draft token of 40 tiles: 8 sub-ranges of 5 tiles, one per lane
    # (each lane's sub-range may itself be cut where the lane groups' ranges meet)
    segs = check([1], [40 * 128], 152, 8)
    per_lane = {}
    for s in segs:
        lo, hi = per_lane.get(s[1], (s[4], s[5]))
        per_lane[s[1]] = (min(lo, s[4]), max(hi, s[5]))
    assert [per_lane[r] for r in range(8)] == [(5 * i, 5 * i + 5) for i in range(8)]
    # 3 column groups on 8 lanes: 2 sub-ranges each, lanes 6 and 7 idle
    segs = check([3], [20 * 128], 152, 8)
    assert {s[1] for s in segs} == set(range(6))


def test_long_token_is_cut_into_at_most_64_pieces():
    # one request far longer than the others: C grows so that it has <= 64 partials
    for w in (1, 2, 4, 8):
        check([1, 1], [64 * 128 * 200, 128], 152, w)
        check([2], [128 * 10000], 152, w)
