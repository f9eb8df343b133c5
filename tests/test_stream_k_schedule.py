"""CPU check of the stream-K schedule invariants the fixed-owner hand-off relies on
(moe_hm_gemm_gb300/csrc/hm_sched.cuh, used by the tcgen05 kernels and the decode kernel): the
(tile, k-block) space is cut into G contiguous ranges, start(c) = floor(c * total / G); the owner of a
split tile (the CTA holding its first k-block) meets it as the last segment of its range, every
other contributor meets it as its first segment and publishes at most one partial, and the
publishers of a tile are exactly the CTAs after its owner up to the one holding its last k-block.
Both grids the planner makes are covered: tiles cut into equal K ranges (G = tiles x floor(SMs /
tiles), when tiles <= SMs) and ranges running across tile boundaries (G = min(SMs, units)).
Test infrastructure, no GPU."""
import random

import pytest


def sk_start(c, total, g):
    return c * total // g


def sk_owner(it, total, g):
    """CTA whose range holds iteration `it` (the same search as the device code)."""
    c = it * g // total
    while c + 1 < g and sk_start(c + 1, total, g) <= it:
        c += 1
    while c > 0 and sk_start(c, total, g) > it:
        c -= 1
    return c


def check(tiles, kb, grid):
    total = tiles * kb
    publishers = {}
    for c in range(grid):
        u0, u1 = sk_start(c, total, grid), sk_start(c + 1, total, grid)
        assert u1 > u0, "every CTA holds at least one k-block"
        segs = []
        for u in range(u0, u1):
            t, k = divmod(u, kb)
            if segs and segs[-1][0] == t:
                segs[-1][2] = k + 1
            else:
                segs.append([t, k, k + 1])
        published = 0
        for i, (t, a, b) in enumerate(segs):
            if a == 0 and b == kb:
                continue                               # a whole tile: no hand-off
            lo, hi = sk_owner(t * kb, total, grid), sk_owner(t * kb + kb - 1, total, grid)
            assert lo < hi
            if c == lo:
                assert a == 0 and i == len(segs) - 1, "the owner meets its split tile last"
            else:
                assert a > 0 and i == 0, "a contributor meets the split tile first"
                published += 1
                publishers.setdefault(t, set()).add(c)
        assert published <= 1
    for t, cs in publishers.items():
        lo, hi = sk_owner(t * kb, total, grid), sk_owner(t * kb + kb - 1, total, grid)
        assert cs == set(range(lo + 1, hi + 1))


def grids(tiles, kb, sms):
    units = tiles * kb
    out = {min(sms, units)}                           # ranges across tile boundaries
    if tiles <= sms:
        out.add(tiles * min(sms // tiles, kb))        # equal K ranges per tile
    return sorted(out)


CASES = [(32, 32), (112, 32), (32, 112), (1, 1), (1, 200), (2, 1), (200, 1), (152, 1), (8, 8), (7, 13),
         (160, 8), (76, 3)]
_rng = random.Random(1)
CASES += [(_rng.randint(1, 300), _rng.randint(1, 120)) for _ in range(120)]


@pytest.mark.parametrize("tiles,kb", CASES)
def test_fixed_owner_invariants(tiles, kb):
    for sms in (1, 2, 3, 148, 152, 160):
        for g in grids(tiles, kb, sms):
            check(tiles, kb, g)


def test_equal_ranges_align_with_clusters():
    """When the grid is a multiple r of the tiles, CTAs r t .. r t + r - 1 hold exactly tile t (so
    the decode kernel may form a thread-block cluster of them), whatever the k-block count."""
    for tiles, kb, r in ((76, 3, 2), (38, 5, 4), (32, 32, 4), (64, 7, 2)):
        g, total = tiles * r, tiles * kb
        for c in range(g):
            u0, u1 = sk_start(c, total, g), sk_start(c + 1, total, g)
            assert u0 // kb == c // r and (u1 - 1) // kb == c // r
