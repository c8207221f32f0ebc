"""Host restatement of the TMA decode kernel's work partition, checked for the
invariants its merge relies on (no GPU).

The kernel lays the sequences' attended 16-position slabs end to end on a
virtual line on which sequence s occupies [P_s + U s, P_s + U s + U + n_s)
(P_s: attended slabs before it, n_s: its own), the first U positions standing
for the cost of a unit.  CTA j of a kv head takes the real slabs of the
virtual range [j c, (j + 1) c), c = max(ceil((S + U N) / R), ceil(max_n /
(kmax - 1)), 1).  A row's merge counts its CTAs as np = floor((v + n - 1) /
c) - floor(v / c) + 1 and its own slot as j - floor(v / c), v = P_s + U (s +
1) the virtual position of the row's first slab.  These must hold for any
lengths: the CTAs' real ranges tile [0, S) in order, a row's slabs are
covered by exactly np consecutive CTAs whose slots are 0 .. np - 1, and np
never exceeds the workspace's kmax slots.
"""
import random

import pytest


def _real(v, P, n, U):
    """Real slab index of virtual position v (v inside the line)."""
    for s in range(len(n)):
        vp = P[s] + U * s
        if vp <= v < vp + U + n[s]:
            return P[s] + min(max(v - vp - U, 0), n[s])
    raise AssertionError("position past the line")


def _ranges(n, R, U, kmax):
    P = [sum(n[:s]) for s in range(len(n))]
    total = sum(n)
    totalv = total + U * len(n)
    cpc = (totalv + R - 1) // R
    if kmax > 1:
        cpc = max(cpc, (max(n) + kmax - 2) // (kmax - 1))
    cpc = max(cpc, 1)
    out = []
    for j in range(R):
        v0, v1 = j * cpc, min(j * cpc + cpc, totalv)
        x0 = _real(v0, P, n, U) if v0 < totalv else total
        x1 = _real(v1, P, n, U) if v1 < totalv else total
        out.append((x0, x1))
    return P, total, cpc, out


@pytest.mark.parametrize("U", [0, 8, 48, 200])
def test_ranges_tile_the_slabs_and_rows_count_their_ctas(U):
    rng = random.Random(1234 + U)
    for _ in range(400):
        N = rng.randint(1, 40)
        n = [rng.choice([0, rng.randint(1, 300), rng.randint(1, 20)]) for _ in range(N)]
        if sum(n) == 0:
            n[0] = 1
        R = rng.randint(1, 40)
        kmax = rng.choice([0, 2, 3, 8, 64])
        P, total, cpc, ranges = _ranges(n, R, U, kmax)
        # the ranges tile [0, total) in CTA order
        pos = 0
        for x0, x1 in ranges:
            assert x0 <= x1
            if x0 < total:
                assert x0 == pos
            pos = max(pos, x1)
        assert pos == total
        for s in range(N):
            if n[s] == 0:
                continue
            covering = [j for j, (x0, x1) in enumerate(ranges) if x0 < P[s] + n[s] and x1 > P[s]]
            v = P[s] + U * (s + 1)
            np_ = (v + n[s] - 1) // cpc - v // cpc + 1
            assert len(covering) == np_
            assert [j - v // cpc for j in covering] == list(range(np_))
            if kmax > 1:
                assert np_ <= kmax


def test_weighting_moves_slabs_away_from_ctas_with_more_sequences():
    # one long sequence and many short ones: without weighting every CTA
    # takes the same slab count; with it the CTAs over the short sequences
    # (more units each) take fewer slabs than those inside the long one
    n = [2000] + [40] * 50
    _, _, _, flat = _ranges(n, 10, 0, 0)
    _, _, _, weighted = _ranges(n, 10, 48, 0)
    sizes_flat = [x1 - x0 for x0, x1 in flat]
    sizes_w = [x1 - x0 for x0, x1 in weighted]
    assert max(sizes_flat) - min(sizes_flat) <= 1
    assert sizes_w[0] > sizes_w[-1]
    assert sum(sizes_w) == sum(n)
