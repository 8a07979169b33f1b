"""Pins of the L2 model oracle: the first page's predicted hit rates and
Spearman values, plus hand-traced cache behaviour (CPU only)."""
import pytest

from conftest import read_lines
from oracle import l2_model as l2
from oracle import tile_order as to


def _fixture():
    rows, cfg, spear = [], None, {}
    for ln in read_lines("tbs_l2_model_8192.txt"):
        if ln[0] == "config":
            cfg = {ln[i]: int(ln[i + 1]) for i in range(1, len(ln), 2)}
        elif ln[0] == "spearman":
            spear[ln[1]] = float(ln[2])
        else:
            rows.append((int(ln[0]), int(ln[1]), float(ln[2]), float(ln[3]),
                         float(ln[4]), float(ln[5]), float(ln[6])))
    return cfg, rows, spear


def test_lru_by_hand():
    c = l2.ByteLRU(capacity_bytes=20)
    # A(10) B(10) fit; A hit refreshes A; C(10) evicts B (oldest); B misses
    # again and evicts A; C hits.
    trace = [("A", 10), ("B", 10), ("A", 10), ("C", 10), ("B", 10), ("C", 10), ("A", 10)]
    got = [c.touch(k, b) for k, b in trace]
    assert got == [False, False, True, False, False, True, False]
    assert (c.hits, c.misses) == (2, 5)


def test_lru_keeps_one_oversized_entry():
    c = l2.ByteLRU(capacity_bytes=5)
    assert not c.touch("X", 50)
    assert c.touch("X", 50)          # still held although above budget
    assert not c.touch("Y", 50)       # X evicted, Y held alone
    assert not c.touch("X", 50)


def test_unbounded_cache_only_compulsory_misses():
    gm, gn, gk = 6, 7, 5
    tiles = to.tile_sequence(to.PANEL, gm, gn, 3)
    c = l2.simulate(tiles, gk, 100, 300, 10**12, concurrency=4)
    assert c.misses == gm * gk + gn * gk
    assert c.miss_bytes == gm * gk * 100 + gn * gk * 300  # compulsory bytes
    assert c.hits == 2 * gm * gn * gk - c.misses


def test_zero_cache_hits_only_on_immediate_reuse():
    # a cache that keeps one tile: consecutive A and B accesses alternate, so
    # nothing is ever re-touched immediately -> no hits
    tiles = to.tile_sequence(to.ROW, 3, 3)
    c = l2.simulate(tiles, 2, 10, 10, 0, concurrency=3)
    assert c.hits == 0


@pytest.mark.slow
def test_printed_predicted_hit_rates():
    cfg, rows, _ = _fixture()
    for order, g, pct, *_ in rows:
        got = l2.predict_l2_hit_rate(order, cfg["M"], cfg["N"], cfg["K"], cfg["bm"],
                                     cfg["bn"], cfg["bk"], cfg["l2_mib"],
                                     cfg["concurrency"], cfg["elem_bytes"], group=g)
        assert round(got, 2) == pytest.approx(pct, abs=1e-9), (order, g, got)


def test_printed_spearman():
    _, rows, spear = _fixture()
    pred = [r[2] for r in rows]
    assert round(l2.rank_correlation(pred, [r[4] for r in rows]), 3) == spear["nonpersistent"]
    assert round(l2.rank_correlation(pred, [r[6] for r in rows]), 3) == spear["persistent"]


def test_spearman_closed_forms():
    assert l2.rank_correlation([1, 2, 3, 4], [10, 20, 30, 40]) == pytest.approx(1.0)
    assert l2.rank_correlation([1, 2, 3, 4], [4, 3, 2, 1]) == pytest.approx(-1.0)
    # ties are not averaged: equal values take their stable-sort positions
    assert l2.rank_correlation([5, 5, 5], [1, 2, 3]) == pytest.approx(1.0)
    assert l2.rank_correlation([2, 1, 1], [3, 1, 2]) == pytest.approx(1.0)
    # a single pair has zero rank variance
    assert l2.rank_correlation([1.0], [2.0]) == 0.0


def test_cluster_cta_sequence():
    seq = l2.cta_tiles_of_clusters(to.PANEL, 4, 3, 2, cluster_m=2)
    # cluster grid 2 x 3 walked group-major with G=2 (= col-major here)
    assert seq[:6] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1), (1, 1)]
    assert sorted(seq) == [(m, n) for m in range(4) for n in range(3)]


def test_k_alternate_by_hand():
    # two waves of one tile each, (0, 0) then (0, 1), four K steps, a cache
    # of two 1-byte tiles.  Ascending in both waves, the second wave finds
    # nothing: 16 misses.  With the second wave descending it starts on
    # A(0, 3), the line the first wave touched last but one: a hit; then
    # B(3, 1) evicts B(3, 0), A(0, 2) evicts A(0, 3), and everything else
    # misses: 1 hit, 15 misses.
    tiles = [(0, 0), (0, 1)]
    up = l2.simulate(tiles, 4, 1, 1, 2, concurrency=1)
    assert (up.hits, up.misses) == (0, 16)
    alt = l2.simulate(tiles, 4, 1, 1, 2, concurrency=1, k_alternate=True)
    assert (alt.hits, alt.misses) == (1, 15)


def test_k_alternate_leaves_first_wave_and_compulsory_misses():
    tiles = to.tile_sequence(to.SERPENTINE, 6, 7, 2)
    # one wave: nothing descends
    a = l2.simulate(tiles, 5, 100, 300, 4000, concurrency=len(tiles))
    b = l2.simulate(tiles, 5, 100, 300, 4000, concurrency=len(tiles), k_alternate=True)
    assert (a.hits, a.misses) == (b.hits, b.misses)
    # an unbounded cache: still only the compulsory misses
    c = l2.simulate(tiles, 5, 100, 300, 10**12, concurrency=4, k_alternate=True)
    assert c.misses == 6 * 5 + 7 * 5
    # one K step: the direction does not matter
    d = l2.simulate(tiles, 1, 100, 300, 500, concurrency=4)
    e = l2.simulate(tiles, 1, 100, 300, 500, concurrency=4, k_alternate=True)
    assert (d.hits, d.misses) == (e.hits, e.misses)


def test_k_alternate_reuses_across_waves():
    # row order, one row of 8 tiles in waves of 2: the A tiles of row 0 are
    # shared by every wave; with the K direction alternating, each wave
    # starts on the A tile the previous wave touched last and hits it
    tiles = to.tile_sequence(to.ROW, 1, 8)
    gk, cap = 6, 3
    up = l2.simulate(tiles, gk, 1, 1, cap, concurrency=2)
    alt = l2.simulate(tiles, gk, 1, 1, cap, concurrency=2, k_alternate=True)
    assert up.hits == 4 * gk  # within a wave only: the second tile's A
    assert alt.hits == up.hits + 3  # plus one A tile at each of 3 wave boundaries
