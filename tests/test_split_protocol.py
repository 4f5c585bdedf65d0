"""The split-tile protocol of the stream-K kernels, checked on the CPU.

Every kernel numbers its units tile-major and gives CTA b the contiguous
range [b U / B, (b+1) U / B).  A tile whose units fall in more than one
range is finished by its first contributor bf; the others publish one
partial sum each (in their slot 0) and count themselves in, and bf waits
for nc - 1 arrivals.  That is only correct if, for every launch shape:

* the tile is bf's last tile and bf's part is the end of its range (bf
  comes to it last and never publishes it);
* for every other contributor the tile is its first tile and its part is
  the start of its range (so it publishes at most once, into slot 0, and
  early);
* the contributor count and first contributor that each kernel works out
  from its own range (cta_of, the first / last tile formulas) equal the
  real ones.

This test recomputes the contributors of every split tile by brute force
from the unit ranges and compares them with those formulas, written as the
kernels write them, over launch shapes of the tests, the benchmark and
larger grids."""
import pytest


def cta_start(b, U, B):
    return b * U // B


def cta_of(u, U, B):
    b = u * B // U
    while b + 1 < B and cta_start(b + 1, U, B) <= u:
        b += 1
    while b > 0 and cta_start(b, U, B) > u:
        b -= 1
    return b


def kernel_view(b, U, B, G):
    """What CTA b works out (the kernels' epilogue set-up): its first and
    last tile, and for each of them whether it is split, its first
    contributor and its contributor count."""
    u0, u1 = cta_start(b, U, B), cta_start(b + 1, U, B)
    tile_first, tile_last = u0 // G, (u1 - 1) // G
    bfA, ncA, ncZ = b, 1, 1
    ts, te = tile_first * G, tile_first * G + G
    if u0 > ts or u1 < te:
        bfA = cta_of(ts, U, B)
        ncA = cta_of(te - 1, U, B) - bfA + 1
    tz = tile_last * G
    if tile_last != tile_first and u1 < tz + G:
        ncZ = cta_of(tz + G - 1, U, B) - b + 1
    view = {}
    for tile in range(tile_first, tile_last + 1):
        s, e = tile * G, tile * G + G
        split = not (u0 <= s and u1 >= e)
        first = tile == tile_first
        view[tile] = (split, bfA if first else b, ncA if first else ncZ)
    return u0, u1, view


def check_shape(U, B, G):
    ranges = [(cta_start(b, U, B), cta_start(b + 1, U, B)) for b in range(B)]
    assert all(u1 > u0 for u0, u1 in ranges), "every CTA has work (B <= U)"
    # brute force: contributors of every tile that a CTA boundary splits
    contrib = {}
    for b, (u0, u1) in enumerate(ranges):
        for tile in range(u0 // G, (u1 - 1) // G + 1):
            contrib.setdefault(tile, []).append(b)
    publishes = [0] * B
    finishes = [0] * B
    for tile, cs in contrib.items():
        if len(cs) == 1:
            continue
        bf, nc = cs[0], len(cs)
        assert cs == list(range(bf, bf + nc)), "contiguous contributors"
        s, e = tile * G, tile * G + G
        u0, u1 = ranges[bf]
        assert (u1 - 1) // G == tile and u1 < e, "the tile is bf's last and its part ends bf's range"
        finishes[bf] += 1
        for c in cs[1:]:
            v0, v1 = ranges[c]
            assert v0 // G == tile and v0 > s, "the tile is the contributor's first; its part starts its range"
            publishes[c] += 1
        # every contributor's own view agrees
        for c in cs:
            _, _, view = kernel_view(c, U, B, G)
            split, vbf, vnc = view[tile]
            assert split, (tile, c)
            assert vbf == bf, (tile, c, vbf, bf)
            if c == bf:
                assert vnc == nc, (tile, c, vnc, nc)
    assert max(publishes) <= 1 and max(finishes) <= 1
    # tiles a CTA sees as complete really have one contributor
    for b in range(B):
        _, _, view = kernel_view(b, U, B, G)
        for tile, (split, _, _) in view.items():
            assert split == (len(contrib[tile]) > 1), (b, tile)


# units per tile G: the 64-row kernel (one unit per 128-column group: K =
# 512 .. 17,408), the tcgen05 kernel (two groups per unit), the 512-row
# kernel (one group)
SHAPES = []
for G in (4, 8, 20, 40, 68, 136):
    for tiles in (1, 2, 3, 7, 40, 80, 151, 152, 153, 160, 304, 544, 640, 1940, 3880):
        for B in (152, 148, 160, 16):
            U = tiles * G
            SHAPES.append((U, min(B, U), G))


@pytest.mark.parametrize("U,B,G", SHAPES)
def test_split_tile_invariants(U, B, G):
    check_shape(U, B, G)


def test_the_check_catches_a_wrong_contributor_count():
    """Not vacuous: an off-by-one in the last tile's count is reported."""
    global kernel_view
    orig = kernel_view

    def bad_view(b, U, B, G):
        u0, u1, view = orig(b, U, B, G)
        return u0, u1, {t: (s, bf, nc + (1 if t == (u1 - 1) // G and nc > 1 else 0)) for t, (s, bf, nc) in view.items()}
    kernel_view = bad_view
    try:
        with pytest.raises(AssertionError):
            check_shape(40 * 136, 152, 136)
    finally:
        kernel_view = orig
