"""Host-side check of the split kernel's work plan (no GPU).

The plan is restated here in Python from its rules:

- each token has tiles_b = ceil(L_b / 128) key tiles plus SEG_COST empty units (the cost
  of a segment's start and end), so request b has T_b * (tiles_b + SEG_COST) units;
- units are numbered request by request, token by token, tile by tile;
- split CTA k owns units [k C, (k + 1) C), with C = max(ceil(U / grid),
  ceil(max_tiles / 63), min(max_tiles, 3) + SEG_COST, 1), and skips the empty units;
- CTA k writes the partial of token index tok (row minus qo_indptr[0]) to segment slot
  tok + k;
- the merge of a token reads slots tok + k0 .. tok + k0 + nseg - 1.

The test walks every CTA's range as the kernel does and checks:

- every unit is covered exactly once;
- each token's pieces come from CTAs k0 .. k0 + nseg - 1, and those are the slots its
  merge reads;
- no two partials share a slot;
- the slots stay below total_q + grid, the workspace's slot count;
- no token is cut into more than 64 pieces, nor into more than ceil(tiles / C) + 1.
"""
import math
import random

import pytest

TILE = 128
NSPLIT = 64
SEG_COST = 1


def plan(T, L, grid):
    tiles = [math.ceil(l / TILE) if t > 0 else 0 for t, l in zip(T, L)]
    cum = [0]
    for t, n in zip(T, tiles):
        cum.append(cum[-1] + t * (n + SEG_COST))
    U = cum[-1]
    maxt = max([n for n, t in zip(tiles, T) if t > 0], default=0)
    C = max(math.ceil(U / grid), math.ceil(maxt / (NSPLIT - 1)), min(maxt, 3) + SEG_COST, 1)
    return tiles, cum, U, C


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


def walk(T, tiles, cum, U, C, grid):
    """Every CTA's segments: (k, b, t, first unit, end unit, slot)."""
    qbase = [0]
    for t in T:
        qbase.append(qbase[-1] + t)
    segs = []
    for k in range(grid):
        u, u_end = k * C, min(U, (k + 1) * C)
        while u < u_end:
            b = unit_request(cum, u)
            per = tiles[b] + SEG_COST
            off = u - cum[b]
            t, j0 = divmod(off, per)
            if j0 >= tiles[b]:          # the token's empty units
                u = cum[b] + (t + 1) * per
                continue
            end = min(u_end, cum[b] + t * per + tiles[b])
            assert end > u
            segs.append((k, b, t, u, end, qbase[b] + t + k))
            u = end
    return segs, qbase


def check(T, L, grid):
    tiles, cum, U, C = plan(T, L, grid)
    assert C * grid >= U
    segs, qbase = walk(T, tiles, cum, U, C, grid)
    covered = [0] * U
    by_token = {}
    for k, b, t, u0, u1, slot in segs:
        for u in range(u0, u1):
            covered[u] += 1
        by_token.setdefault((b, t), []).append((k, u0, u1, slot))
    # every key tile covered once, every empty unit never
    for b in range(len(T)):
        for t in range(T[b]):
            base = cum[b] + t * (tiles[b] + SEG_COST)
            for u in range(base, base + tiles[b]):
                assert covered[u] == 1
            for u in range(base + tiles[b], base + tiles[b] + SEG_COST):
                assert covered[u] == 0
    used = set()
    total_q = qbase[-1]
    for (b, t), pieces in by_token.items():
        pieces.sort()
        u0 = cum[b] + t * (tiles[b] + SEG_COST)
        assert pieces[0][1] == u0 and pieces[-1][2] == u0 + tiles[b]
        k0, k1 = u0 // C, (u0 + tiles[b] - 1) // C
        nseg = k1 - k0 + 1
        assert nseg == len(pieces) and nseg <= NSPLIT
        assert nseg <= math.ceil(tiles[b] / C) + 1
        assert [pc[0] for pc in pieces] == list(range(k0, k1 + 1))
        tok = qbase[b] + t
        if nseg > 1:
            assert [pc[3] for pc in pieces] == [tok + k for k in range(k0, k1 + 1)]
            for _, _, _, sl in pieces:
                assert 0 <= sl < total_q + grid
                assert sl not in used
                used.add(sl)


@pytest.mark.parametrize("seed", range(60))
def test_random_plans(seed):
    rng = random.Random(seed)
    bs = rng.randint(1, 40)
    max_q = rng.randint(1, 16)
    T = [rng.randint(0, max_q) for _ in range(bs)]
    L = [rng.randint(1, 6000) + t for t in T]
    grid = rng.choice([1, 2, 7, 31, 152])
    check(T, L, grid)


def test_bench_like_shapes():
    rng = random.Random(7)
    check([16] * 8, [rng.randint(1024, 4096) + 16 for _ in range(8)], 152)
    check([16], [185000 + 16], 152)
    check([8] * 32, [int(math.exp(rng.uniform(math.log(512), math.log(32768)))) + 8
                     for _ in range(32)], 152)
    T = [rng.choice([1, 4, 8, 16]) for _ in range(64)]
    check(T, [rng.randint(8192, 65536) + t for t in T], 152)
    check([4], [132], 152)


def test_small_batch_is_not_spread_one_tile_per_cta():
    # four drafts of two tiles each on 152 CTAs: C = 2 + SEG_COST, so every token stays whole
    tiles, cum, U, C = plan([4], [132], 152)
    assert C == 2 + SEG_COST
    segs, _ = walk([4], tiles, cum, U, C, 152)
    assert len(segs) == 4 and all(u1 - u0 == 2 for _, _, _, u0, u1, _ in segs)


def test_long_token_is_cut_into_at_most_64_pieces():
    # one request far longer than the others: C grows so that it has <= 64 partials
    check([1, 1], [64 * 128 * 200, 128], 152)
    check([2], [128 * 10000], 152)
