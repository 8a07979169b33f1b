"""Offline L2 hit-rate model and rank correlation (oracle).

Source: Lei Mao, "CUDA Thread Block Swizzle", section "CUDA Thread Block
Swizzle Benchmark": the byte-capacity LRU cache, the wave-by-wave tile trace
and the Spearman rank correlation of predicted hit rate against measured
throughput.

The model, restated:
  * The cache holds whole operand tiles.  Capacity is a byte budget.  A hit
    refreshes the tile's recency.  A miss inserts the tile, then the least
    recently used tiles are dropped while the bytes held exceed the budget and
    more than one tile is held (so a tile larger than the budget still stays).
  * The tile order is evaluated once for every program id.  Consecutive
    ``concurrency`` ids form a wave.  Inside a wave, for every K step in turn,
    each tile of the wave (in id order) touches its A tile (m, k) and then its
    B tile (k, n).
  * Hit rate = hits / (hits + misses), in percent.

``simulate(..., k_alternate=True)`` is not the page's model but the K order
of the library's persistent GEMM: the tiles of every other wave (waves 1, 3,
5, ...) step through K from the last step to the first, the others from the
first to the last.  Everything else is the page's model.
"""
from __future__ import annotations

import math
from collections import OrderedDict

from . import tile_order as to


class ByteLRU:
    """Least-recently-used set of keys with a byte budget."""

    def __init__(self, capacity_bytes):
        self.capacity = capacity_bytes
        self._held = OrderedDict()  # key -> bytes, oldest first
        self.bytes_held = 0
        self.hits = 0
        self.misses = 0
        self.miss_bytes = 0  # bytes brought in by misses: the predicted DRAM reads

    def touch(self, key, nbytes):
        held = self._held
        if key in held:
            self.hits += 1
            held.move_to_end(key)
            return True
        self.misses += 1
        self.miss_bytes += nbytes
        held[key] = nbytes
        self.bytes_held += nbytes
        while self.bytes_held > self.capacity and len(held) > 1:
            _, dropped = held.popitem(last=False)
            self.bytes_held -= dropped
        return False

    def hit_rate_pct(self):
        n = self.hits + self.misses
        return 100.0 * self.hits / n if n else 0.0


def simulate(tiles, grid_k, a_tile_bytes, b_tile_bytes, capacity_bytes,
             concurrency, k_alternate=False):
    """Replay the wave trace of ``tiles`` (a list of (m, n) in program-id
    order) through a ByteLRU.  Returns the cache (hits, misses inside).
    ``k_alternate``: odd waves take the K steps in descending order."""
    cache = ByteLRU(capacity_bytes)
    for w0 in range(0, len(tiles), concurrency):
        wave = tiles[w0:w0 + concurrency]
        descending = k_alternate and (w0 // concurrency) % 2 == 1
        for k in (range(grid_k - 1, -1, -1) if descending else range(grid_k)):
            for m, n in wave:
                cache.touch(("A", m, k), a_tile_bytes)
                cache.touch(("B", k, n), b_tile_bytes)
    return cache


def predict_l2_hit_rate(order, M, N, K, block_m, block_n, block_k,
                        l2_mib, concurrency, elem_bytes, group=1):
    """Predicted L2 hit rate (percent) of one tile order on an M x N x K GEMM
    with block_m x block_n x block_k tiles, an ``l2_mib`` MiB cache and
    ``concurrency`` simultaneously running tiles."""
    gm = math.ceil(M / block_m)
    gn = math.ceil(N / block_n)
    gk = math.ceil(K / block_k)
    tiles = to.tile_sequence(order, gm, gn, group)
    cache = simulate(tiles, gk, block_m * block_k * elem_bytes,
                     block_k * block_n * elem_bytes, l2_mib * 1024 * 1024,
                     concurrency)
    return cache.hit_rate_pct()


def cta_tiles_of_clusters(order, gm, gn, group, cluster_m):
    """CTA-tile sequence induced by a cluster-level order: cluster work w maps
    to cluster tile (mc, n); its CTAs take rows mc*cluster_m + r, r = 0 ..
    cluster_m-1, in rank order ("ClusterPersistentScheduler2D", Example 2)."""
    if gm % cluster_m:
        raise ValueError("cluster_m must divide gm")
    seq = []
    for mc, n in to.tile_sequence(order, gm // cluster_m, gn, group):
        for r in range(cluster_m):
            seq.append(to.cta_tile(mc, n, r, cluster_m, 1))
    return seq


def rank_correlation(xs, ys):
    """Spearman rank correlation as the benchmark computes it: each value's
    rank is its position after a stable ascending sort (ties are not
    averaged), then the Pearson correlation of the two rank vectors; 0 when
    either rank vector has zero variance."""
    def positions(v):
        r = [0] * len(v)
        for pos, i in enumerate(sorted(range(len(v)), key=lambda i: v[i])):
            r[i] = pos
        return r

    rx, ry = positions(xs), positions(ys)
    n = len(xs)
    mx, my = sum(rx) / n, sum(ry) / n
    sxy = sum((a - mx) * (b - my) for a, b in zip(rx, ry))
    sxx = sum((a - mx) ** 2 for a in rx)
    syy = sum((b - my) ** 2 for b in ry)
    if sxx == 0 or syy == 0:
        return 0.0
    return sxy / math.sqrt(sxx * syy)
