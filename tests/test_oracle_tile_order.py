"""Pins of the tile-order oracle against the pages' tables, closed forms and
hand-derived cases (CPU only)."""
import random

import pytest

from conftest import read_lines, read_table
from oracle import tile_order as to


@pytest.mark.parametrize("fname,order,group", [
    ("tbs_row_major_8x8.txt", to.ROW, 1),
    ("tbs_panel_g4_8x8.txt", to.PANEL, 4),
    ("tbs_morton_8x8.txt", to.MORTON, 1),
    ("tbs_xor_8x8.txt", to.XOR, 1),
])
def test_8x8_tables(fname, order, group):
    assert to.id_table(order, 8, 8, group) == read_table(fname)


def test_col_major_is_transposed_row_major():
    # closed form: tile (m, n) is reached by id n*gm + m
    for gm, gn in [(8, 8), (3, 5), (5, 3), (1, 7)]:
        t = to.id_table(to.COL, gm, gn)
        assert t == [[n * gm + m for n in range(gn)] for m in range(gm)]
    row = read_table("tbs_row_major_8x8.txt")
    assert to.id_table(to.COL, 8, 8) == [list(r) for r in zip(*row)]


def test_group_major_table_equals_panel():
    assert to.id_table(to.PANEL, 4, 4, 2) == read_table("cps_group_major_4x4_g2.txt")


def test_serpentine_table():
    assert to.id_table(to.SERPENTINE, 4, 4, 2) == read_table("cps_serpentine_4x4_s2.txt")


def test_panel_degenerate_groups():
    # G = 1 walks rows (row-major); G >= gm is one band walked down columns.
    for gm, gn in [(8, 8), (6, 10), (5, 3)]:
        assert to.tile_sequence(to.PANEL, gm, gn, 1) == to.tile_sequence(to.ROW, gm, gn)
        for g in (gm, gm + 3):
            assert to.tile_sequence(to.PANEL, gm, gn, g) == to.tile_sequence(to.COL, gm, gn)


def test_panel_ragged_last_band_by_hand():
    # 5 x 3 grid, G = 2: bands of rows {0,1}, {2,3} and the 1-row tail {4}.
    assert to.id_table(to.PANEL, 5, 3, 2) == [
        [0, 2, 4], [1, 3, 5], [6, 8, 10], [7, 9, 11], [12, 13, 14]]


def test_serpentine_degenerate_and_ragged():
    for gm, gn in [(4, 4), (3, 7), (6, 2)]:
        # one strip as wide as the grid: row-major
        assert to.tile_sequence(to.SERPENTINE, gm, gn, gn) == to.tile_sequence(to.ROW, gm, gn)
        # strips one tile wide: columns walked alternately down and up
        assert to.id_table(to.SERPENTINE, gm, gn, 1) == [
            [n * gm + (m if n % 2 == 0 else gm - 1 - m) for n in range(gn)]
            for m in range(gm)]
    # 3 x 5 grid, S = 2: strips {0,1} down, {2,3} up, tail strip {4} down
    assert to.id_table(to.SERPENTINE, 3, 5, 2) == [
        [0, 1, 10, 11, 12], [2, 3, 8, 9, 13], [4, 5, 6, 7, 14]]


def test_morton_xor_bijective_on_square_powers_of_two():
    # the first page: both are bijective for power-of-two (square) grids
    for e in range(0, 7):
        g = 1 << e
        assert to.is_bijective(to.MORTON, g, g)
        assert to.is_bijective(to.XOR, g, g)


def test_morton_not_bijective_by_hand():
    # 3 x 3: id 5 has bits 0b101 -> m = 0b11 = 3 -> 3 mod 3 = 0, n = 0: tile
    # (0, 0) again, already taken by id 0.
    assert to.morton(5, 3, 3) == (0, 0) == to.morton(0, 3, 3)
    assert not to.is_bijective(to.MORTON, 3, 3)


def test_xor_not_bijective_by_hand():
    # 2 x 4 grid: id 0 -> x=0,y=0 -> (0,0); id 2 -> x=2,y=0 -> (2 mod 2, 0) = (0,0)
    assert to.xor_swizzle(0, 2, 4) == to.xor_swizzle(2, 2, 4) == (0, 0)
    assert not to.is_bijective(to.XOR, 2, 4)


def test_panel_and_serpentine_always_bijective():
    rnd = random.Random(1)
    for _ in range(60):
        gm, gn, g = rnd.randint(1, 23), rnd.randint(1, 23), rnd.randint(1, 9)
        assert to.is_bijective(to.PANEL, gm, gn, g)
        assert to.is_bijective(to.SERPENTINE, gm, gn, g)
        assert to.is_bijective(to.ROW, gm, gn)
        assert to.is_bijective(to.COL, gm, gn)


def _three_cluster_fixture():
    lines = read_lines("cps_three_clusters.txt")
    owner, work, seq, cta = [], {}, {}, []
    mode = None
    for ln in lines:
        if ln[0] == "owner":
            mode = "owner"
        elif ln[0] == "work":
            work[int(ln[1])] = [int(v) for v in ln[2:]]
        elif ln[0] == "seq":
            v = [int(x) for x in ln[2:]]
            seq[int(ln[1])] = list(zip(v[0::2], v[1::2]))
        elif ln[0] == "cta":
            cta.append([int(x) for x in ln[1:]])
        elif mode == "owner":
            owner.append([int(x) for x in ln])
    return owner, work, seq, cta


def test_three_cluster_distribution():
    owner, work, seq, _ = _three_cluster_fixture()
    seqs = to.cluster_sequences(4, 4, 3, to.PANEL, 2)
    for c in range(3):
        assert [w for w, _, _ in seqs[c]] == work[c]
        assert [(m, n) for _, m, n in seqs[c]] == seq[c]
        for _, m, n in seqs[c]:
            assert owner[m][n] == c


def test_scheduler_state_machine():
    s = to.ClusterSchedule(4, 4, 3, to.PANEL, 2)
    s.init(2)
    assert (s.work_idx, s.tile_count, s.m_idx, s.n_idx) == (2, 0, 0, 1)
    s.next_tile()
    assert (s.work_idx, s.tile_count, s.m_idx, s.n_idx) == (5, 1, 1, 2)
    s.next_tile_stride(100)
    assert not s.valid() and s.tile_count == 2


def test_cta_split_example():
    *_, cta = _three_cluster_fixture()
    for m_idx, n_idx, rank, cm, cn in cta:
        assert to.cta_tile(m_idx, n_idx, rank, 2, 1) == (cm, cn)


def test_persistent_trace_closed_forms():
    gm, gn = 6, 5
    for order, g in [(to.ROW, 1), (to.PANEL, 4), (to.SERPENTINE, 2)]:
        ids = {mn: p for p, mn in enumerate(to.tile_sequence(order, gm, gn, g))}
        # non-persistent: program p takes tile id p, once
        tr = to.persistent_trace(order, gm, gn, g, gm * gn)
        assert tr == {mn: (p, 0) for mn, p in ids.items()}
        # persistent with P programs: id p runs on program p mod P at step p div P
        P = 7
        tr = to.persistent_trace(order, gm, gn, g, P)
        assert tr == {mn: (p % P, p // P) for mn, p in ids.items()}
    # 2-CTA clusters on a 6 x 5 CTA grid = 3 x 5 cluster grid, 4 clusters
    cids = {mn: w for w, mn in enumerate(to.tile_sequence(to.PANEL, 3, 5, 2))}
    tr = to.persistent_trace(to.PANEL, 6, 5, 2, 8, cluster_m=2)
    assert len(tr) == 30
    for (cm, n), (prog, it) in tr.items():
        w = cids[(cm // 2, n)]
        assert prog == 2 * (w % 4) + cm % 2 and it == w // 4


def test_persistent_trace_2x2_clusters():
    # [CPS] Example 2 with cluster_m = cluster_n = 2: a 6 x 8 CTA grid is a
    # 3 x 4 cluster grid; rank r of a cluster owns CTA tile (2m + r mod 2,
    # 2n + r div 2) of cluster tile (m, n)
    cids = {mn: w for w, mn in enumerate(to.tile_sequence(to.SERPENTINE, 3, 4, 2))}
    P = 12  # 3 clusters
    tr = to.persistent_trace(to.SERPENTINE, 6, 8, 2, P, cluster_m=2, cluster_n=2)
    assert len(tr) == 48
    for (cm, cn), (prog, it) in tr.items():
        w = cids[(cm // 2, cn // 2)]
        assert prog == 4 * (w % 3) + (cm % 2) + 2 * (cn % 2) and it == w // 3
    # hand-derived: serpentine S=2 on the 3 x 4 cluster grid, id 1 = cluster
    # tile (0, 1); cluster 1 takes it first (iteration 0); CTA tile (1, 2) is
    # its row 1, column 0 -> rank 1 -> program 4 + 1
    assert tr[(1, 2)] == (5, 0)
    assert tr[(0, 3)] == (6, 0)   # rank 2 of cluster 1: row 0, column 1
    with pytest.raises(ValueError):
        to.persistent_trace(to.ROW, 6, 7, 1, 4, cluster_m=2, cluster_n=2)


def test_stream_k_trace_hand_example():
    # 1 x 3 tiles, 4 clusters, 4 K blocks a tile: all 3 tiles are the tail,
    # I = 12 blocks split [0,3) [3,6) [6,9) [9,12).  Tile 0 starts at block 0
    # (cluster 0, its first item); tile 1 at block 4, inside cluster 1's
    # range, whose items are the end of tile 0 (item 0) and tile 1 (item 1);
    # tile 2 at block 8, cluster 2's second item.  Cluster 3 only adds the
    # end of tile 2.
    assert to.stream_k_ranges(4, 3, 4) == [(0, 3), (3, 6), (6, 9), (9, 12)]
    assert to.stream_k_trace(to.ROW, 1, 3, 1, 4, 4) == {
        (0, 0): (0, 0), (0, 1): (1, 1), (0, 2): (2, 1)}
    # the same with 2-CTA clusters: each cluster tile is two CTA tiles
    assert to.stream_k_trace(to.ROW, 2, 3, 1, 8, 4, cluster_m=2) == {
        (0, 0): (0, 0), (1, 0): (1, 0), (0, 1): (2, 1), (1, 1): (3, 1),
        (0, 2): (4, 1), (1, 2): (5, 1)}
    with pytest.raises(ValueError):
        to.stream_k_trace(to.ROW, 3, 3, 1, 8, 4, cluster_m=2)


def test_stream_k_trace_hand_example_with_whole_units():
    # 1 x 5 tiles in row order, 3 clusters, 2 K blocks a tile.  Units 0-2 go
    # out whole (one per cluster); units 3 and 4 are the tail: I = 4 blocks,
    # ranges [0,1) [1,2) [2,4).  The tail pieces come first: cluster 0 holds
    # block 0, the head of unit 3 (its item 0), cluster 1 block 1 (the end of
    # unit 3), cluster 2 blocks 2-3, all of unit 4 (its item 0); each
    # cluster's whole unit is its item 1.
    assert to.stream_k_ranges(3, 2, 2) == [(0, 1), (1, 2), (2, 4)]
    assert to.stream_k_trace(to.ROW, 1, 5, 1, 3, 2) == {
        (0, 0): (0, 1), (0, 1): (1, 1), (0, 2): (2, 1), (0, 3): (0, 0), (0, 4): (2, 0)}
    # 1 x 4 tiles, 3 clusters, 1 K block a tile: one tail unit, I = 1 block,
    # ranges [0,0) [0,0) [0,1): clusters 0 and 1 have no tail piece, so their
    # whole units are their items 0; cluster 2 takes the tail unit first
    assert to.stream_k_ranges(3, 1, 1) == [(0, 0), (0, 0), (0, 1)]
    assert to.stream_k_trace(to.ROW, 1, 4, 1, 3, 1) == {
        (0, 0): (0, 0), (0, 1): (1, 0), (0, 2): (2, 1), (0, 3): (2, 0)}


@pytest.mark.parametrize("gm,gn,P,kb,cm", [(6, 5, 6, 4, 1), (6, 5, 7, 16, 1), (6, 5, 7, 3, 1),
                                           (6, 5, 40, 3, 1), (2, 1, 152, 16384, 2),
                                           (6, 5, 8, 9, 2), (10, 4, 6, 7, 2)])
def test_stream_k_trace_against_brute_force(gm, gn, P, kb, cm):
    order, g = to.PANEL, 2
    tr = to.stream_k_trace(order, gm, gn, g, P, kb, cluster_m=cm)
    assert len(tr) == gm * gn  # every CTA tile written once
    clusters, U = P // cm, (gm // cm) * gn
    R = U % clusters
    if R == 0:
        assert tr == to.persistent_trace(order, gm, gn, g, P, cluster_m=cm)
        return
    # the tail, block by block: owner of block b = the cluster whose range
    # holds it; ranges are contiguous, cover [0, R * kb) once and differ in
    # length by at most one block
    ranges = to.stream_k_ranges(clusters, R, kb)
    # whole units: as the static schedule, after the cluster's tail pieces
    seq = to.tile_sequence(order, gm // cm, gn, g)
    for w in range(U - R):
        m, n = seq[w]
        c = w % clusters
        npieces = len({b // kb for b in range(*ranges[c])})
        for r in range(cm):
            assert tr[(m * cm + r, n)] == (c * cm + r, npieces + w // clusters)
    assert ranges[0][0] == 0 and ranges[-1][1] == R * kb
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    assert max(e - s for s, e in ranges) - min(e - s for s, e in ranges) <= 1
    holder = {}
    for c, (s, e) in enumerate(ranges):
        for b in range(s, e):
            holder[b] = c
    for t in range(R):
        c = holder[t * kb]
        # the items of cluster c before this one: one per earlier tail unit
        # its range touches
        earlier = len({b // kb for b in range(*ranges[c]) if b // kb < t})
        m, n = seq[U - R + t]
        for r in range(cm):
            assert tr[(m * cm + r, n)] == (c * cm + r, earlier)


def test_die_split_trace_hand_example():
    # 1 x 6 tiles in row order, 4 clusters on dies 0, 1, 1, 0: P0 = 2, so die
    # 0 takes U0 = floor((6 * 2 + 2) / 4) = 3 units.  Die 0's clusters 0 and 3
    # (ranks 0, 1) stride over units 0-2, die 1's clusters 1 and 2 over 3-5.
    dies = [0, 1, 1, 0]
    assert to.die_split_trace(to.ROW, 1, 6, 1, dies) == {
        (0, 0): (0, 0), (0, 1): (3, 0), (0, 2): (0, 1),
        (0, 3): (1, 0), (0, 4): (2, 0), (0, 5): (1, 1)}
    # with a Stream-K tail, 2 K blocks a tile: each die has 3 units on 2
    # clusters, so units 0, 1 (die 0) and 3, 4 (die 1) go out whole and units
    # 2 and 5 are split block by block ([0,1) and [1,2)); the first block's
    # cluster holds the head (its item 0), whole units come after the pieces
    assert to.die_split_trace(to.ROW, 1, 6, 1, dies, k_blocks=2) == {
        (0, 0): (0, 1), (0, 1): (3, 1), (0, 2): (0, 0),
        (0, 3): (1, 1), (0, 4): (2, 1), (0, 5): (1, 0)}
    # 2-CTA clusters: each cluster tile is two CTA tiles, programs 2g and 2g+1
    tr = to.die_split_trace(to.ROW, 2, 6, 1, dies, cluster_m=2)
    assert tr[(0, 1)] == (6, 0) and tr[(1, 1)] == (7, 0) and tr[(1, 5)] == (3, 1)


@pytest.mark.parametrize("gm,gn,P,kb,cm", [(6, 5, 6, None, 1), (6, 5, 7, 4, 1), (8, 7, 10, 3, 2),
                                           (4, 3, 9, 5, 1), (2, 1, 12, 64, 2)])
def test_die_split_trace_covers_every_tile_once(gm, gn, P, kb, cm):
    import random
    rnd = random.Random(gm * 100 + P)
    for _ in range(5):
        dies = [rnd.randint(0, 1) for _ in range(P)]
        tr = to.die_split_trace(to.SERPENTINE, gm, gn, 2, dies, k_blocks=kb, cluster_m=cm)
        assert len(tr) == gm * gn
        # a program's item indices are 0, 1, 2, ... without gaps over its whole
        # units (its tail pieces come before, and only heads are recorded)
        for prog in range(P * cm):
            its = sorted(it for p, it in tr.values() if p == prog)
            assert len(set(its)) == len(its)
    # every cluster on one die: the plain schedules
    assert to.die_split_trace(to.PANEL, 6, 5, 2, [0] * 7) == to.persistent_trace(to.PANEL, 6, 5, 2, 7)
    assert to.die_split_trace(to.PANEL, 6, 5, 2, [1] * 7, k_blocks=3) == to.stream_k_trace(
        to.PANEL, 6, 5, 2, 7, 3)
