"""Host-side pins of the sparse GEMM's stream-K partition (no GPU).

Stream-K gives CTA pair c of P the k-steps [c T / P, (c + 1) T / P) of all T = tiles x nk steps in tile-major
order ("RT-Lynx" page, Method, CUDA kernel optimisation: the page splits its sparse GEMM's work stream-K
fashion).  The kernel keeps kPairMaxSplit = 4 partial slots per tile, and the host enables the schedule only where
tiles >= P / 2 and nk >= 8.  These tests restate the partition and check, over the whole range the host allows,
that it covers every k-step of every tile exactly once, that the parts of a tile are numbered in k order by
the pair that owns each step, and that no tile has more than four parts."""
import pytest


def owner(step, P, T):
    """The pair whose range holds k-step `step`: the last c with floor(c T / P) <= step."""
    return ((step + 1) * P - 1) // T


def units(c, P, tiles, nk):
    """Pair c's units in order: (tile, kbeg, kend, part, parts)."""
    T = tiles * nk
    b0, b1 = c * T // P, (c + 1) * T // P
    out = []
    t = b0 // nk
    while b0 < b1 and t * nk < b1:
        kbeg = max(b0 - t * nk, 0)
        kend = min(b1 - t * nk, nk)
        first = owner(t * nk, P, T)
        out.append((t, kbeg, kend, c - first, owner(t * nk + nk - 1, P, T) - first + 1))
        t += 1
    return out


def test_owner_is_the_range_start_rule():
    P, T = 7, 100
    starts = [c * T // P for c in range(P + 1)]
    for s in range(T):
        c = owner(s, P, T)
        assert starts[c] <= s < starts[c + 1]


@pytest.mark.parametrize("P", [4, 7, 38, 74, 76])
def test_partition_covers_every_step_once_in_at_most_four_parts(P):
    worst = 0
    for tiles in range(-(-P // 2), 3 * P + 2):
        for nk in (8, 9, 13, 24, 48, 96):
            parts = {}
            for c in range(P):
                for t, kb, ke, part, nparts in units(c, P, tiles, nk):
                    assert 0 <= kb < ke <= nk
                    parts.setdefault(t, []).append((kb, ke, part, nparts))
            assert sorted(parts) == list(range(tiles))
            for t, ps in parts.items():
                ps.sort()
                assert ps[0][0] == 0 and ps[-1][1] == nk
                for i, (kb, ke, part, nparts) in enumerate(ps):
                    assert part == i and nparts == len(ps)
                    if i:
                        assert ps[i - 1][1] == kb
                worst = max(worst, len(ps))
    assert worst <= 4


def test_fewer_tiles_than_half_the_pairs_can_need_more_parts():
    """Why the host requires tiles >= P / 2: with fewer tiles a tile can span five or more pairs' ranges."""
    P, tiles, nk = 76, 8, 96
    most = max(nparts for c in range(P) for *_, nparts in units(c, P, tiles, nk))
    assert most > 4


def stagger(mp, nb, num_mp, nk_u):
    """The producer's staggered k order for a two-row-block tile: pair (mp, nb) starts at offset
    ((mp + nb) mod G) * min(nk_u, 24) / G, G = min(8, num_mp), and wraps around."""
    G = min(8, num_mp)
    rot = ((mp + nb) % G) * min(nk_u, 24) // G
    return [(it + rot) % nk_u for it in range(nk_u)], rot


def test_stagger_is_a_permutation_of_the_unit_steps():
    for num_mp in (1, 2, 3, 8, 9, 32):
        for nk_u in (1, 2, 7, 24, 25, 96):
            for mp in range(num_mp):
                for nb in range(10):
                    order, rot = stagger(mp, nb, num_mp, nk_u)
                    assert 0 <= rot < nk_u or nk_u == 1 and rot == 0
                    assert sorted(order) == list(range(nk_u))


def test_stagger_separates_the_pairs_that_share_a_column_tile():
    """The pairs of one W column tile (same nb, consecutive mp) start on different k-steps when there are up to
    eight of them and at least eight steps."""
    for num_mp in (2, 4, 8, 9, 36):
        for nk_u in (8, 24, 96):
            for nb in range(5):
                starts = [stagger(mp, nb, num_mp, nk_u)[1] for mp in range(min(num_mp, 8))]
                assert len(set(starts)) == len(starts)
