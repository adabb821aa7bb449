"""A model of how the decode kernel splits a batch's tiles over its CTAs.

Each (sequence, KV head) segment costs PC units for its piece end (a
constant of the kernel's configuration) followed by one unit per work unit
of tiles; the total cost is split evenly over
P = min(grid, cost) CTAs and a CTA owns the tiles whose cost position falls
in its share.  The kernel finds a CTA's first and last tile from the cost
prefix in one pass, and the owner of a tile (for the cross-CTA merge counts)
from the tile's cost position.  This model restates both computations and
checks, over random length mixes (empty sequences, one-tile segments, long
ones), that:

* the CTAs' tile ranges partition the tiles in order;
* the owner computed from a tile's cost position is the CTA whose range
  holds it;
* every CTA from the owner of a segment's first tile to the owner of its
  last tile holds a tile of that segment (the merge waits for exactly that
  many partials).

No GPU is involved.
"""
import random


def owner_of(x, total, parts):
    return ((x + 1) * parts - 1) // total


def split(nts, hkv, pc, grid):
    ts, cs = [0], [0]
    for nt in nts:
        ts.append(ts[-1] + nt * hkv)
        cs.append(cs[-1] + ((nt + pc) * hkv if nt > 0 else 0))
    T, CT = ts[-1], cs[-1]
    P = min(grid, CT)
    ranges = []
    for c in range(grid):
        bounds = []
        for cb in ((c * CT // P, (c + 1) * CT // P) if c < P else (CT, CT)):
            r = T
            for b, nt in enumerate(nts):             # the sequence whose cost holds cb
                cost = (nt + pc) * hkv if nt > 0 else 0
                if cs[b] <= cb < cs[b] + cost:
                    rem = cb - cs[b]
                    kvh = rem // (nt + pc)
                    inn = rem - kvh * (nt + pc) - pc
                    r = ts[b] + kvh * nt + min(max(inn, 0), nt)
            bounds.append(r)
        ranges.append(tuple(bounds))
    return ts, cs, T, CT, P, pc, ranges


def test_split_invariants():
    for trial in range(1500):
        rng = random.Random(trial)
        B = rng.randint(1, 30)
        hkv = rng.choice([1, 2, 4, 8])
        pc = rng.choice([1, 2, 6, 10, 16, 18])
        grid = rng.choice([1, 2, 5, 16, 152])
        nts = [rng.choice([0, 0, 1, 2, 3, 5, 17, 100, 400]) for _ in range(B)]
        ts, cs, T, CT, P, pc, ranges = split(nts, hkv, pc, grid)
        if T == 0:
            continue
        # a partition in order
        assert ranges[0][0] == 0 and ranges[-1][1] == T
        for c in range(grid - 1):
            assert ranges[c][1] == ranges[c + 1][0]
        own = {}
        for c, (r0, r1) in enumerate(ranges):
            assert r0 <= r1
            for x in range(r0, r1):
                own[x] = c
        for b, nt in enumerate(nts):
            for kvh in range(hkv if nt else 0):
                first = cs[b] + kvh * (nt + pc) + pc
                for i in range(nt):
                    assert owner_of(first + i, CT, P) == own[ts[b] + kvh * nt + i]
                c0, c1 = owner_of(first, CT, P), owner_of(first + nt - 1, CT, P)
                holders = {own[ts[b] + kvh * nt + i] for i in range(nt)}
                assert holders == set(range(c0, c1 + 1))


def test_split_charges_piece_ends():
    # 8 long sequences and 64 one-tile ones: CTAs that take the short ones
    # take fewer tiles than an even split of tiles would give them
    nts = [400] * 8 + [1] * 64
    ts, cs, T, CT, P, pc, ranges = split(nts, 8, 18, 16)
    sizes = [r1 - r0 for r0, r1 in ranges]
    assert max(sizes) > T // 16 > min(sizes)
