"""Host-side check of the fused shard-sum GEMM's tile schedule (gemm.cuh: fused_tile, and the unit
count of launch_gemm_t for that variant), restated here: units walk output tiles unit, unit + units,
... while whole rounds remain; a last round that would keep at most half the units busy is split into
half-width tiles, two per tile; a launch with at most half as many tiles as the device's CTA pairs
gets two units per tile.  For every tile count and device size: every column of every output tile is
produced by exactly one unit, a half-width tile's two halves go to two different units, and no unit
is given more rounds than the busiest one needs."""
import pytest


def units_for(tiles, max_units):
    want = 2 * tiles if 2 * tiles <= max_units else tiles
    return min(want, max_units)


def fused_tile(o, tiles, unit, units):
    """(tile, half) of output tile o of a unit, or None past its end; half = -1 for a whole tile."""
    full, rest = divmod(tiles, units)
    split = rest > 0 and 2 * rest <= units
    if o < full or (o == full and not split):
        ot, half = unit + o * units, -1
    else:
        if o > full or unit >= 2 * rest:
            return None
        ot, half = full * units + (unit >> 1), unit & 1
    return None if ot >= tiles else (ot, half)


@pytest.mark.parametrize("max_units", [1, 2, 3, 7, 38, 76])
def test_every_tile_column_exactly_once(max_units):
    for tiles in range(1, 700):
        units = units_for(tiles, max_units)
        cover = {}
        rounds = []
        for u in range(units):
            o = 0
            while True:
                t = fused_tile(o, tiles, u, units)
                if t is None:
                    break
                ot, half = t
                for h in ((0, 1) if half < 0 else (half,)):
                    assert (ot, h) not in cover, (tiles, units, ot, h)
                    cover[(ot, h)] = u
                o += 1
            rounds.append(o)
        assert set(cover) == {(ot, h) for ot in range(tiles) for h in (0, 1)}, (tiles, units)
        for ot in range(tiles):
            if cover[(ot, 0)] != cover[(ot, 1)]:
                # a split tile: its halves on two units, in the last round only
                assert ot >= (tiles // units) * units
        full, rest = divmod(tiles, units)
        assert max(rounds) == full + (1 if rest else 0)


def test_split_happens_where_it_shortens_the_last_round():
    # 320 output tiles (GPT-3 2.7B second linear, one row chunk) on 76 CTA pairs: 4 whole rounds and
    # 16 tiles split over 32 units; 1024 tiles (Llama-3 8B): 13 rounds and 36 tiles over 72 units
    for tiles, split_units in ((320, 32), (1024, 72)):
        units = units_for(tiles, 76)
        last = [u for u in range(units) if fused_tile(tiles // units, tiles, u, units) is not None]
        assert len(last) == split_units
        assert all(fused_tile(tiles // units, tiles, u, units)[1] in (0, 1) for u in last)
    # 4 tiles on 76 pairs: 8 units, every tile split
    assert units_for(4, 76) == 8
    assert all(fused_tile(0, 4, u, 8)[1] == (u & 1) for u in range(8))
    # a last round of exactly half the units is split, one of more than half is not
    assert fused_tile(1, 114, 75, 76) == (113, 1)
    assert all(fused_tile(1, 115, u, 76) is None or fused_tile(1, 115, u, 76)[1] == -1 for u in range(76))
