"""The balanced split's share arithmetic, restated in Python and checked
against exact integer arithmetic and brute force (no GPU).

CTA c of C takes global key tiles [lo(c), lo(c + 1)) with lo(c) =
floor(c W / C); the kernel computes it as c q + floor(c r / C) with W = q C + r
in 32-bit integers.  A piece of a cut unit finds the shares holding the
unit's first and last tiles by walking from its own share, counts the
non-empty ones, and publishes to slot 2c (its share's first piece) or 2c + 1.
"""
import random

import pytest

INT32_MAX = (1 << 31) - 1


def lo_exact(c, C, W):
    return (c * W) // C


def lo_kernel(c, C, W):
    q, r = W // C, W % C
    assert c * q <= INT32_MAX and c * r <= INT32_MAX, "32-bit overflow"
    return c * q + (c * r) // C


@pytest.mark.parametrize("seed", range(5))
def test_share_bounds_match_exact_division(seed):
    rng = random.Random(seed)
    for _ in range(2000):
        C = rng.choice([1, 2, 151, 152, 304, 608, rng.randint(1, 46340)])
        W = rng.choice([0, 1, C - 1, C, C + 1, rng.randint(0, INT32_MAX)])
        W = max(W, 0)
        for c in (0, 1, C // 2, C - 1, C):
            assert lo_kernel(c, C, W) == lo_exact(c, C, W)


def pieces(units, C):
    """Brute force: every share's pieces as (unit, first local tile, tiles),
    from the per-unit tile counts laid end to end."""
    W = sum(units)
    start = [0]
    for n in units:
        start.append(start[-1] + n)
    out = []
    for c in range(C):
        a, b = lo_exact(c, C, W), lo_exact(c + 1, C, W)
        ps = []
        for u, n in enumerate(units):
            s, e = max(a, start[u]), min(b, start[u] + n)
            if s < e:
                ps.append((u, s - start[u], e - s))
        out.append(ps)
    return out, start, W


def walk_for_piece(c, gu, n_all, C, W):
    """The kernel's walk: shares c0..c1 holding the unit's first and last
    tiles, the non-empty ones among them, and each one's slot."""
    c0 = c1 = c
    while lo_kernel(c0, C, W) > gu:
        c0 -= 1
    while lo_kernel(c1 + 1, C, W) <= gu + n_all - 1:
        c1 += 1
    shares = [x for x in range(c0, c1 + 1) if lo_kernel(x + 1, C, W) > lo_kernel(x, C, W)]
    slots = {x: 2 * x + (0 if lo_kernel(x, C, W) >= gu else 1) for x in shares}
    return shares, slots


@pytest.mark.parametrize("seed", range(20))
def test_walk_finds_every_piece_of_a_cut_unit(seed):
    rng = random.Random(100 + seed)
    nunits = rng.randint(1, 60)
    units = [rng.randint(1, 40) for _ in range(nunits)]
    C = rng.choice([1, 3, 7, 16, 64, 152, 304])
    per_share, start, W = pieces(units, C)
    owner_of = {}
    for c, ps in enumerate(per_share):
        for k, (u, t0, n) in enumerate(ps):
            owner_of.setdefault(u, []).append((c, k, t0, n))
    for u, lst in owner_of.items():
        if len(lst) == 1:
            assert lst[0][2] == 0 and lst[0][3] == units[u]  # a whole piece
            continue
        expect = sorted(c for c, _, _, _ in lst)
        for c, k, t0, n in lst:
            # every piece of the cut unit recomputes the same share set
            shares, slots = walk_for_piece(c, start[u], units[u], C, W)
            assert shares == expect
            # slot 2c for a share's first piece, 2c + 1 for any later one
            assert slots[c] == 2 * c + (0 if k == 0 else 1)
            # only a share's first piece can start inside a unit, and only its
            # last can end inside one
            if t0 > 0:
                assert k == 0
            if t0 + n < units[u]:
                assert k == len(per_share[c]) - 1
        # the pieces tile the unit exactly once
        covered = sorted((t0, n) for _, _, t0, n in lst)
        pos = 0
        for t0, n in covered:
            assert t0 == pos
            pos += n
        assert pos == units[u]


def test_shares_are_balanced():
    """Shares differ by at most one tile, whatever the unit sizes."""
    for C in (1, 5, 152, 304):
        for W in (0, 1, C - 1, C, 10 * C + 3, 32256):
            sizes = [lo_exact(c + 1, C, W) - lo_exact(c, C, W) for c in range(C)]
            assert sum(sizes) == W
            assert max(sizes) - min(sizes) <= 1
