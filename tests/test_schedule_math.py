"""The split-sequence schedule's arithmetic, checked on the host (no GPU).

The decode kernel cuts every unit (sequence, KV head, head chunk) into
64-token tiles, lays all tiles out as one flat list of N tiles and gives
block c the range [N*c/P, N*(c+1)/P).  A unit cut by range boundaries is
finished by a split combine that relies on three facts, restated here from
the kernel's formulas and checked over many length mixes:

* the block owning tile x is ((x+1)*P - 1) // N (the kernel computes each
  unit's first and last covering block this way);
* with P <= N every block between those two owns a tile of the unit, so the
  unit's arrival count is last - first + 1;
* the partial slot cta + u of every (block, cut unit) pair is distinct and
  below grid + units (the scratch the host allocates).

Equal-length batches may use a unit-aligned P; the last test checks that
such a P puts every range boundary on a unit boundary (or splits every unit
into equal parts).
"""
import random

import pytest


def ranges(N, P):
    return [(N * c // P, N * (c + 1) // P) for c in range(P)]


def block_of_tile(x, N, P):
    return ((x + 1) * P - 1) // N


def units_layout(tiles_per_unit):
    starts, s = [], 0
    for t in tiles_per_unit:
        starts.append(s)
        s += t
    return starts, s


def check_schedule(tiles_per_unit, grid):
    starts, N = units_layout(tiles_per_unit)
    if N == 0:
        return
    P = min(grid, N)
    rg = ranges(N, P)
    assert rg[0][0] == 0 and rg[-1][1] == N
    for c in range(P - 1):
        assert rg[c][1] == rg[c + 1][0]
    # the closed form agrees with the ranges
    for c, (a, b) in enumerate(rg):
        assert b > a  # P <= N: no empty range
        for x in (a, b - 1):
            assert block_of_tile(x, N, P) == c
    slots = set()
    for u, (us, nt) in enumerate(zip(starts, tiles_per_unit)):
        if nt == 0:
            continue
        cf = block_of_tile(us, N, P)
        cl = block_of_tile(us + nt - 1, N, P)
        for c in range(cf, cl + 1):
            a, b = rg[c]
            assert max(a, us) < min(b, us + nt), (u, c)  # owns a tile
        if cf != cl:
            for c in range(cf, cl + 1):
                slot = c + u
                assert slot not in slots
                assert slot < grid + len(tiles_per_unit)
                slots.add(slot)


@pytest.mark.parametrize("seed", range(40))
def test_ragged_batches(seed):
    rnd = random.Random(seed)
    B = rnd.randint(1, 70)
    hu = rnd.choice([1, 2, 8])
    lens = [rnd.randint(0, 3000) for _ in range(B)]
    tiles = []
    for L in lens:
        tiles += [(L + 63) // 64] * hu
    check_schedule(tiles, rnd.choice([1, 7, 64, 148, 296]))


@pytest.mark.parametrize("units,nt,grid", [
    (64, 128, 148),   # 70B shape: units cut across blocks
    (128, 36, 148),   # 8B shape
    (32, 64, 148),    # MQA shape
    (2048, 64, 148),  # MHA shape: many units per block
    (1, 2, 148),      # fewer tiles than blocks
    (3, 1, 2),
])
def test_uniform_batches(units, nt, grid):
    check_schedule([nt] * units, grid)


def test_unit_aligned_block_counts_cut_on_unit_boundaries():
    # P = units (one unit a block), P dividing units, or P = k * units
    # (each unit in k equal parts, +-1 tile)
    for units, nt, P in [(128, 36, 128), (256, 64, 128), (32, 64, 128),
                         (64, 128, 128), (40, 10, 20)]:
        N = units * nt
        rg = ranges(N, P)
        bounds = {b for _, b in rg}
        if P <= units:
            assert units % P == 0
            assert all(b % nt == 0 for b in bounds)
        else:
            k = P // units
            assert P == k * units
            for u in range(units):
                own = [b - a for a, b in rg[u * k:(u + 1) * k]]
                assert sum(own) == nt and max(own) - min(own) <= 1
                assert rg[u * k][0] == u * nt
        check_schedule([nt] * units, P)
