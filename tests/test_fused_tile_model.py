"""Host-side check of the fused shard-sum GEMM's work split (gemm.cuh: fused_tile, tile_at and the
unit count of launch_gemm_t for that variant), restated here.  Units walk output tiles unit,
unit + units, ... while whole rounds remain, each tile with all t shards in order.  A last round of
at most half as many tiles as units (or every tile, when there are fewer tiles than units) is shared
by s = min(t, units // rest) units per tile when the scratch holds its slots: unit u < rest * s takes
shards [i t // s, (i + 1) t // s) of tile u // s, i = u % s, writes each shard's partial to slot
(u // s) * t + g, and i = 0 (the head) then adds slots 0 .. t-1 in order and writes Y.  For every
tile count, shard count and device size: every (tile, shard) product is computed exactly once, every
tile's Y is written exactly once, from its shards in order, each slot is written by one unit and
read by the tile's head, and no unit runs more rounds of sub-tiles than the split needs."""
import pytest

SLOT = 256 * 256 * 4


def launch(tiles, t, max_units, part_bytes):
    """(units, split) as launch_gemm_t chooses them."""
    units = min(tiles, max_units)
    if t > 1 and tiles < max_units:
        units = min(tiles * t, max_units)
    rest = tiles % units
    split = min(t, units // rest) if rest > 0 else 1
    slots = rest * t
    if split >= 2 and part_bytes >= slots * (SLOT + 4):
        return units, split
    if tiles < units:
        units = tiles
    return units, 1


def fused_tile(o, tiles, t, unit, units, split):
    """(tile, lo, hi, role, slot0) or None; role 'whole', 'head' or 'helper'."""
    full, rest = divmod(tiles, units)
    if o < full or (o == full and split <= 1):
        ot = o * units + unit
        if ot >= tiles:
            return None
        return ot, 0, t, "whole", 0
    if o > full or unit >= rest * split:
        return None
    j, i = divmod(unit, split)
    return full * units + j, i * t // split, (i + 1) * t // split, "head" if i == 0 else "helper", j * t


def tile_at(sub, tiles, t, unit, units, split):
    """(tile, shard) of the unit's sub-tile `sub` (the producer's and MMA issuer's order), or None."""
    full = tiles // units
    o = sub // t if sub < full * t else full
    f = fused_tile(o, tiles, t, unit, units, split)
    if f is None:
        return None
    g = f[1] + (sub - o * t)
    return None if g >= f[2] else (f[0], g)


def host_split_bytes(tiles, t, units=76):
    """fused_split_bytes of the API's workspace plan."""
    if tiles == 0 or t < 2:
        return 0
    u = min(tiles * t, units) if tiles < units else units
    rest = tiles % u
    if rest == 0 or u // rest < 2:
        return 0
    return rest * t * (SLOT + 4)


@pytest.mark.parametrize("max_units", [1, 2, 3, 7, 38, 76])
@pytest.mark.parametrize("t", [1, 2, 3, 5, 8])
def test_every_product_once_and_every_y_once_in_order(max_units, t):
    for tiles in range(1, 400):
        units, split = launch(tiles, t, max_units, part_bytes=1 << 40)
        done, y_writers, slot_writer = {}, {}, {}
        rounds = []
        for u in range(units):
            # the epilogue's walk: whole tiles, then the unit's share of a split tile
            full, rest = divmod(tiles, units)
            nwhole = full + (1 if (split <= 1 and u < rest) else 0)
            seq = []
            for o in range(nwhole):
                ot, lo, hi, role, _ = fused_tile(o, tiles, t, u, units, split)
                assert role == "whole" and (lo, hi) == (0, t)
                seq += [(ot, g) for g in range(t)]
                y_writers.setdefault(ot, []).append((u, list(range(t))))
            f = fused_tile(full, tiles, t, u, units, split) if split > 1 else None
            if f is not None:
                ot, lo, hi, role, slot0 = f
                assert lo < hi
                seq += [(ot, g) for g in range(lo, hi)]
                for g in range(lo, hi):
                    assert slot0 + g not in slot_writer
                    slot_writer[slot0 + g] = (u, ot, g)
                if role == "head":
                    y_writers.setdefault(ot, []).append((u, [("slot", slot0 + g) for g in range(t)]))
            # the producer / MMA order is the same
            k = 0
            while (x := tile_at(k, tiles, t, u, units, split)) is not None:
                assert x == seq[k], (tiles, t, u, k)
                k += 1
            assert k == len(seq)
            for x in seq:
                assert x not in done, (tiles, t, u, x)
                done[x] = u
            rounds.append(len(seq))
        assert set(done) == {(ot, g) for ot in range(tiles) for g in range(t)}, (tiles, t, units)
        assert set(y_writers) == set(range(tiles))
        for ot, w in y_writers.items():
            assert len(w) == 1, (tiles, t, ot, w)
            _, order = w[0]
            if order and isinstance(order[0], tuple):
                # the head reads slot g for shard g, in order, each written by some unit of this tile
                assert [slot_writer[s][1:] for _, s in order] == [(ot, g) for g in range(t)]
        full, rest = divmod(tiles, units)
        if split > 1:
            assert rest * split <= units and slot_writer
            assert max(slot_writer) < rest * t
            assert max(rounds) == full * t + max(hi - lo for lo, hi in
                                                  ((i * t // split, (i + 1) * t // split) for i in range(split)))
        else:
            assert max(rounds) == (full + (1 if rest else 0)) * t


def test_split_where_the_last_round_is_short():
    # GPT-3 2.7B second linear, one row chunk: 320 tiles on 76 CTA pairs, t = 8: 4 whole rounds, the
    # last 16 tiles on 64 units with 2 shards each
    assert launch(320, 8, 76, 1 << 40) == (76, 4)
    # Llama-3 8B: 1024 tiles: 13 rounds, 36 tiles on 72 units with 4 shards each
    assert launch(1024, 8, 76, 1 << 40) == (76, 2)
    # a last round of more than half the units is not split
    assert launch(115, 8, 76, 1 << 40) == (76, 1)
    # fewer tiles than units: every tile split, up to one shard per unit
    assert launch(4, 8, 76, 1 << 40) == (32, 8)
    assert launch(20, 8, 76, 1 << 40) == (76, 3)
    # no scratch, or a single shard: no split, no idle units
    assert launch(4, 8, 76, 0) == (4, 1)
    assert launch(320, 1, 76, 1 << 40) == (76, 1)


def test_host_workspace_matches_the_launcher_on_76_pairs():
    for tiles in range(1, 2000):
        for t in (1, 2, 4, 8):
            need = host_split_bytes(tiles, t)
            units, split = launch(tiles, t, 76, need)
            if need:
                assert split > 1, (tiles, t)
            else:
                assert split == 1
            # with exactly the planned bytes the launcher splits whenever it would with unlimited scratch
            assert launch(tiles, t, 76, 1 << 40)[1] == split


def unit_subtiles(tiles, t, unit, units, split):
    """gemm.cuh unit_subtiles for the fused shard-sum (the MMA issuer's count)."""
    full, rest = divmod(tiles, units)
    if split <= 1:
        return (full + (1 if unit < rest else 0)) * t
    if unit >= rest * split:
        return full * t
    i = unit % split
    return full * t + (i + 1) * t // split - i * t // split


@pytest.mark.parametrize("max_units", [1, 3, 38, 76])
def test_mma_count_matches_the_sequence(max_units):
    for tiles in range(1, 300):
        for t in (1, 2, 3, 8):
            units, split = launch(tiles, t, max_units, part_bytes=1 << 40)
            for u in range(units):
                k = 0
                while tile_at(k, tiles, t, u, units, split) is not None:
                    k += 1
                assert unit_subtiles(tiles, t, u, units, split) == k, (tiles, t, u)


def test_mma_count_of_the_other_variants():
    # every other variant: tiles unit, unit + units, ... of batches x m_tiles x n_tiles
    for total in range(0, 500):
        for units in (1, 7, 76):
            for u in range(units):
                want = len(range(u, total, units))
                got = (total - 1 - u) // units + 1 if u < total else 0
                assert got == want
