"""Host-side property of the projection GEMM's stream-K split.

The (N tile, M tile, K block) units are cut into contiguous CTA ranges
[c U / C, (c + 1) U / C).  Every CTA that touches output tile t writes one
partial, and the partial buffer holds `maxc` of them per tile, with
maxc = min(C, KB, KB // (U // C) + 2) (C <= U CTAs, KB K blocks a tile).
The kernel relies on no tile having more contributors than that, and the
readers on tile t's contributors being CTAs c0(t)..c1(t) with
c0 = ((t KB + 1) C - 1) // U and c1 = ((t + 1) KB C - 1) // U.  Both are
checked here by brute force over the CTA ranges.
"""
import random

import pytest


def _contributors(U, C, KB):
    tiles = U // KB
    per = [set() for _ in range(tiles)]
    for c in range(C):
        lo, hi = c * U // C, (c + 1) * U // C
        for u in range(lo, hi):
            per[u // KB].add(c)
    return per


def _cases():
    rng = random.Random(7)
    cases = [(32 * 64, 152, 64), (80 * 64, 152, 64), (4 * 32 * 64, 152, 64), (64, 64, 1),
             (20 * 16, 152, 16), (9, 9, 9), (152 * 3, 152, 3), (153, 152, 1)]
    for _ in range(200):
        KB = rng.randint(1, 130)
        tiles = rng.randint(1, 90)
        U = tiles * KB
        C = rng.randint(1, min(U, 160))
        cases.append((U, C, KB))
    return cases


@pytest.mark.parametrize("U,C,KB", _cases())
def test_partial_count_bound_and_contributor_range(U, C, KB):
    per = _contributors(U, C, KB)
    maxc = min(C, KB, KB // (U // C) + 2)
    for t, cs in enumerate(per):
        assert 1 <= len(cs) <= maxc
        c0 = ((t * KB + 1) * C - 1) // U
        c1 = ((t + 1) * KB * C - 1) // U
        assert cs == set(range(c0, c1 + 1))
