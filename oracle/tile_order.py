"""Program-id -> output-tile maps and the cluster-persistent schedule (oracle).

Sources:
  [TBS] Lei Mao, "CUDA Thread Block Swizzle": sections "Linear Swizzle",
        "Grouped 2D Panel Swizzle", "Morton / Z-order Swizzle", "Bitwise XOR
        Swizzle" (8x8 tables) and the benchmark script's CPU mapping functions
        and persistent tile loop.
  [CPS] TVM TIRx docs, "ClusterPersistentScheduler2D": "Tile Ordering"
        (group-major), "Serpentine Mode", "Example 1: Basic persistent kernel",
        "Example 2: 2SM GEMM".

All functions return (m, n): m indexes output-tile rows (the M dimension),
n output-tile columns (N).  The pages' tables print the program id at
(row = m, column = n).
"""
from __future__ import annotations

ROW, COL, PANEL, MORTON, XOR, SERPENTINE = 0, 1, 2, 3, 4, 5
ORDER_NAMES = {ROW: "row", COL: "col", PANEL: "panel", MORTON: "morton",
               XOR: "xor", SERPENTINE: "serpentine"}


def row_major(pid, gm, gn):
    """[TBS] Linear Swizzle: consecutive ids walk along N, then the next row."""
    return pid // gn, pid % gn


def col_major(pid, gm, gn):
    """[TBS] linear column-major mapper: consecutive ids walk along M first."""
    return pid % gm, pid // gm


def panel(pid, gm, gn, group):
    """[TBS] Grouped 2D Panel Swizzle with group size G along M.

    Ids are dealt out group by group; a group is a band of G tile rows spanning
    all gn columns.  Inside a band the ids run down a column of the band first
    (column-major inside the band).  The last band holds only the rows that are
    left (gm - first_row of that band), and that smaller height is the period
    used inside it.  [CPS] "Tile Ordering" (group-major with l2_group_size) is
    the same map.
    """
    ids_per_band = group * gn
    band = pid // ids_per_band
    first_row = band * group
    band_rows = min(gm - first_row, group)
    within = pid - band * ids_per_band
    return first_row + within % band_rows, within // band_rows


def morton(pid, gm, gn):
    """[TBS] Morton / Z-order: bit 2i of the id is bit i of m, bit 2i+1 is bit
    i of n (16 bit pairs), each then reduced modulo its grid extent."""
    m = 0
    n = 0
    for i in range(16):
        m |= ((pid >> (2 * i)) & 1) << i
        n |= ((pid >> (2 * i + 1)) & 1) << i
    return m % gm, n % gn


def xor_swizzle(pid, gm, gn):
    """[TBS] Bitwise XOR: with x = id mod gn and y = id div gn, the tile row is
    (x XOR y) mod gm and the tile column is y mod gn."""
    x = pid % gn
    y = pid // gn
    return (x ^ y) % gm, y % gn


def serpentine(pid, gm, gn, size):
    """[CPS] Serpentine Mode, read from its 4x4 table (swizzle_size = S).

    The N axis is cut into strips S tiles wide.  Strip s is walked one tile row
    at a time, left to right inside the row; even strips go down the rows
    (m = 0 .. gm-1), odd strips go up (m = gm-1 .. 0).  A last strip narrower
    than S (when S does not divide gn) uses its own width as the row length.
    """
    strip = pid // (size * gm)
    r = pid - strip * size * gm
    width = min(size, gn - strip * size)
    step = r // width
    m = step if strip % 2 == 0 else gm - 1 - step
    n = strip * size + r % width
    return m, n


def tile_of(order, pid, gm, gn, group=1):
    """Dispatch on the order id ([TBS] mode ids 0..4; 5 = serpentine)."""
    if order == ROW:
        return row_major(pid, gm, gn)
    if order == COL:
        return col_major(pid, gm, gn)
    if order == PANEL:
        return panel(pid, gm, gn, group)
    if order == MORTON:
        return morton(pid, gm, gn)
    if order == XOR:
        return xor_swizzle(pid, gm, gn)
    if order == SERPENTINE:
        return serpentine(pid, gm, gn, group)
    raise ValueError(f"unknown order {order}")


def tile_sequence(order, gm, gn, group=1):
    """[(m, n) for pid in 0 .. gm*gn-1]."""
    return [tile_of(order, p, gm, gn, group) for p in range(gm * gn)]


def is_bijective(order, gm, gn, group=1):
    """True when the map visits every one of the gm*gn tiles exactly once."""
    seen = set(tile_sequence(order, gm, gn, group))
    if len(seen) != gm * gn:
        return False
    return all(0 <= m < gm and 0 <= n < gn for m, n in seen)


def id_table(order, gm, gn, group=1):
    """gm x gn table whose entry (m, n) is the id mapped to tile (m, n), as
    the pages print it.  Entries never reached stay None."""
    t = [[None] * gn for _ in range(gm)]
    for p, (m, n) in enumerate(tile_sequence(order, gm, gn, group)):
        t[m][n] = p
    return t


class ClusterSchedule:
    """[CPS] cluster-persistent work distribution, restated.

    A cluster starts at work index ``cluster_id`` and advances by
    ``num_clusters``; it is valid while the work index is below the number of
    tiles; the current (m, n) is the tile order applied to the work index;
    ``tile_count`` counts the tiles handed out so far.
    """

    def __init__(self, gm, gn, num_clusters, order=PANEL, group=8):
        self.gm, self.gn = gm, gn
        self.num_clusters = num_clusters
        self.order, self.group = order, group
        self.work_idx = 0
        self.tile_count = 0
        self.m_idx = self.n_idx = 0

    def _update(self):
        if self.valid():
            self.m_idx, self.n_idx = tile_of(self.order, self.work_idx,
                                             self.gm, self.gn, self.group)

    def init(self, cluster_id):
        self.work_idx = cluster_id
        self.tile_count = 0
        self._update()

    def valid(self):
        return self.work_idx < self.gm * self.gn

    def next_tile_stride(self, stride):
        self.work_idx += stride
        self.tile_count += 1
        self._update()

    def next_tile(self):
        self.next_tile_stride(self.num_clusters)


def cluster_sequences(gm, gn, num_clusters, order=PANEL, group=8):
    """For every cluster, its list of (work_idx, m, n) in execution order."""
    out = []
    for c in range(num_clusters):
        s = ClusterSchedule(gm, gn, num_clusters, order, group)
        s.init(c)
        seq = []
        while s.valid():
            seq.append((s.work_idx, s.m_idx, s.n_idx))
            s.next_tile()
        out.append(seq)
    return out


def cta_tile(m_idx, n_idx, cta_idx, cluster_m, cluster_n):
    """[CPS] Example 2: a cluster-level tile becomes per-CTA tiles outside the
    scheduler.  rank = cta_idx mod cluster size; the rank's position inside the
    cluster is (rank mod cluster_m, rank div cluster_m)."""
    rank = cta_idx % (cluster_m * cluster_n)
    cb_m = rank % cluster_m
    cb_n = rank // cluster_m
    return m_idx * cluster_m + cb_m, n_idx * cluster_n + cb_n


def persistent_trace(order, gm, gn, group, num_programs, cluster_m=1, cluster_n=1):
    """What a persistent launch of ``num_programs`` CTAs does, CTA by CTA.

    Programs are grouped into clusters of cluster_m x cluster_n CTAs; the
    scheduler works on the cluster-tile grid (gm / cluster_m) x (gn /
    cluster_n) and every CTA of a cluster takes its own CTA tile of the
    cluster tile ([CPS] Example 2: rank -> (rank mod cluster_m, rank div
    cluster_m)).  With cluster_m = cluster_n = 1 and num_programs = tiles this
    is the non-persistent launch of [TBS] (one program per tile, one loop
    iteration each).

    Returns {(cta_m, cta_n): (program, iteration)} over all CTA tiles.
    """
    if gm % cluster_m or gn % cluster_n:
        raise ValueError("the cluster shape must divide the CTA-tile grid")
    size = cluster_m * cluster_n
    num_clusters = num_programs // size
    seqs = cluster_sequences(gm // cluster_m, gn // cluster_n, num_clusters, order, group)
    trace = {}
    for c, seq in enumerate(seqs):
        for it, (_, m_idx, n_idx) in enumerate(seq):
            for r in range(size):
                prog = c * size + r
                key = cta_tile(m_idx, n_idx, prog, cluster_m, cluster_n)
                if key in trace:
                    raise AssertionError(f"tile {key} visited twice")
                trace[key] = (prog, it)
    return trace


def stream_k_trace(order, gm, gn, group, num_programs, k_blocks, cluster_m=1):
    """The persistent schedule with a Stream-K tail, CTA by CTA.

    Not from the pages: the first page names dynamic balancing and Stream-K
    only as what its static loop lacks.  This is the library's definition,
    written out plainly.  With P clusters of cluster_m CTAs and U
    scheduler units (cluster tiles, in tile-order sequence), the first
    U - R units (R = U mod P) go out whole by work-index striding, as in
    persistent_trace.  The K blocks of the R tail units are laid end to
    end, I = R * k_blocks of them, and cluster c takes the contiguous range
    [floor(I c / P), floor(I (c + 1) / P)).  A cluster's work items are
    first one item for each tail unit its range touches, in K order, then
    its whole units.  A tail unit is recorded for the cluster whose range
    holds the unit's first K block, at that cluster's item for the unit.

    Returns {(cta_m, cta_n): (program, item index)} over all CTA tiles: the
    program and item that write each whole tile, and for a tail tile the
    program and item holding its first K block.
    """
    if gm % cluster_m:
        raise ValueError("the cluster shape must divide the CTA-tile grid")
    seq = tile_sequence(order, gm // cluster_m, gn, group)
    P = num_programs // cluster_m
    U = len(seq)
    R = U % P
    full = U - R
    trace = {}

    def put(unit, c, item):
        m_idx, n_idx = seq[unit]
        for r in range(cluster_m):
            key = (m_idx * cluster_m + r, n_idx)
            if key in trace:
                raise AssertionError(f"tile {key} written twice")
            trace[key] = (c * cluster_m + r, item)

    I = R * k_blocks
    pieces = []  # tail units each cluster's range touches
    for c in range(P):
        s, e = I * c // P, I * (c + 1) // P
        touched = []
        t = s // k_blocks
        while s < e and t * k_blocks < e:
            if t * k_blocks >= s:
                put(full + t, c, len(touched))
            touched.append(t)
            t += 1
        pieces.append(len(touched))
    for w in range(full):
        put(w, w % P, pieces[w % P] + w // P)
    return trace


def stream_k_ranges(num_clusters, tail_units, k_blocks):
    """Each cluster's tail range [s, e) in the laid-end-to-end K blocks."""
    I = tail_units * k_blocks
    return [(I * c // num_clusters, I * (c + 1) // num_clusters)
            for c in range(num_clusters)]


def die_split_trace(order, gm, gn, group, cluster_die, k_blocks=None, cluster_m=1):
    """The persistent schedule with its work split between two dies, CTA by CTA.

    Not from the pages: the library's die split.  Cluster g (CTAs
    g * cluster_m .. g * cluster_m + cluster_m - 1) sits on die
    cluster_die[g] (0 or 1); its rank is the number of clusters before it on
    the same die.  With P clusters, P0 of them on die 0, and U scheduler
    units in tile-order sequence, die 0 takes units [0, U0) and die 1 units
    [U0, U), where U0 = floor((U * P0 + floor(P / 2)) / P), that is U * P0 / P
    rounded with halves going up.  Each die schedules its units over its own
    clusters as a launch of that many clusters would: by work-index striding
    (the die's unit i goes to its rank i mod P_d as that cluster's item
    i div P_d), or, with k_blocks given, with a Stream-K tail of the die's
    own R_d = U_d mod P_d units over its P_d clusters as in stream_k_trace
    (a cluster's tail pieces first, then its whole units).  With every
    cluster on one die the launch is not split.

    Returns {(cta_m, cta_n): (program, item index)} as stream_k_trace.
    """
    if gm % cluster_m:
        raise ValueError("the cluster shape must divide the CTA-tile grid")
    P = len(cluster_die)
    members = [[g for g in range(P) if cluster_die[g] == d] for d in (0, 1)]
    if not members[0] or not members[1]:
        if k_blocks is None:
            return persistent_trace(order, gm, gn, group, P * cluster_m, cluster_m=cluster_m)
        return stream_k_trace(order, gm, gn, group, P * cluster_m, k_blocks, cluster_m)
    seq = tile_sequence(order, gm // cluster_m, gn, group)
    U = len(seq)
    U0 = (U * len(members[0]) + P // 2) // P
    trace = {}

    def put(unit, g, item):
        m_idx, n_idx = seq[unit]
        for r in range(cluster_m):
            key = (m_idx * cluster_m + r, n_idx)
            if key in trace:
                raise AssertionError(f"tile {key} written twice")
            trace[key] = (g * cluster_m + r, item)

    for d, (lo, hi) in enumerate(((0, U0), (U0, U))):
        Pd, Ud = len(members[d]), hi - lo
        R = Ud % Pd if k_blocks is not None else 0
        full = Ud - R
        pieces = [0] * Pd
        if R:
            I = R * k_blocks
            for r in range(Pd):
                s, e = I * r // Pd, I * (r + 1) // Pd
                t = s // k_blocks
                while s < e and t * k_blocks < e:
                    if t * k_blocks >= s:
                        put(lo + full + t, members[d][r], pieces[r])
                    pieces[r] += 1
                    t += 1
        for w in range(full):
            put(lo + w, members[d][w % Pd], pieces[w % Pd] + w // Pd)
    return trace
