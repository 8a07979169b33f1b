"""The library's host L2 model (swz_l2_model) reproduces the oracle's hit and
miss counts exactly (CPU only)."""
import math

import pytest

from conftest import read_lines
from oracle import l2_model as l2
from oracle import tile_order as to


@pytest.fixture(scope="module")
def swz():
    from thread_block_smem_gb300 import build
    build.build()
    import thread_block_smem_gb300 as m
    return m


def _oracle_counts(order, group, M, N, K, tm, tn, tk, eb, l2b, conc, cm, k_alternate=False):
    gm = cm * math.ceil(M / (tm * cm))
    gn = math.ceil(N / tn)
    gk = math.ceil(K / tk)
    seq = l2.cta_tiles_of_clusters(order, gm, gn, group, cm)
    c = l2.simulate(seq, gk, tm * tk * eb, tk * tn * eb, l2b, conc, k_alternate)
    return c.hits, c.misses, c.miss_bytes


CASES = [
    # order, group, M, N, K, tile_m, tile_n, tile_k, elem, l2 bytes, concurrency, cluster_m
    (to.ROW, 1, 1024, 1024, 512, 128, 128, 64, 2, 1 << 20, 16, 1),
    (to.PANEL, 4, 1024, 1024, 512, 128, 128, 64, 2, 1 << 20, 16, 1),
    (to.SERPENTINE, 2, 2048, 1536, 256, 128, 256, 64, 2, 3 << 20, 20, 1),
    (to.PANEL, 8, 4096, 4096, 1024, 128, 256, 64, 2, 8 << 20, 148, 2),
    (to.SERPENTINE, 4, 4096, 4096, 1024, 128, 256, 64, 2, 8 << 20, 152, 2),
    (to.MORTON, 1, 4096, 4096, 1024, 128, 256, 64, 2, 8 << 20, 152, 2),
    (to.XOR, 1, 2048, 2048, 512, 128, 128, 32, 2, 2 << 20, 40, 1),
    (to.COL, 1, 1000, 1200, 300, 128, 128, 64, 4, 1 << 20, 7, 1),
    (to.PANEL, 3, 1000, 1200, 300, 128, 256, 64, 2, 0, 5, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_native_model_matches_oracle(swz, case):
    rc, h, m = swz.swz_l2_model(*case)
    assert rc == 0
    want = _oracle_counts(*case)
    assert (h, m) == want[:2]
    rc, h2, m2, b = swz.swz_l2_model_bytes(*case)
    assert rc == 0 and (h2, m2, b) == want


@pytest.mark.parametrize("parts", [2, 3])
@pytest.mark.parametrize("case", CASES[2:6])
def test_partitioned_model_is_the_oracle_at_a_fraction_of_the_capacity(swz, case, parts):
    # the two-die reading: each of `parts` halves replays the whole trace with
    # 1/parts of the capacity (integer division of the byte budget)
    rc, h, m, b = swz.swz_l2_model_bytes(*case, l2_partitions=parts)
    assert rc == 0
    c = list(case)
    c[9] = case[9] // parts
    assert (h, m, b) == _oracle_counts(*c)


@pytest.mark.parametrize("parts", [1, 2])
@pytest.mark.parametrize("case", CASES)
def test_k_alternate_matches_oracle(swz, case, parts):
    # the persistent GEMM's K order: odd waves descending
    rc, h, m, b = swz.swz_l2_model_bytes(*case, l2_partitions=parts, k_alternate=1)
    assert rc == 0
    c = list(case)
    c[9] = case[9] // parts
    assert (h, m, b) == _oracle_counts(*c, k_alternate=True)


@pytest.mark.slow
def test_native_model_reproduces_printed_rates(swz):
    rows = [ln for ln in read_lines("tbs_l2_model_8192.txt") if ln[0] not in ("config", "spearman")]
    for r in rows:
        order, g, pct = int(r[0]), int(r[1]), float(r[2])
        got = swz.l2_model_hit_rate(order, g, 8192, 8192, 8192, 128, 128, 32, 2,
                                    64 << 20, 168, 1)
        assert round(got, 2) == pytest.approx(pct, abs=1e-9), (order, g, got)


def test_native_miss_bytes_compulsory(swz):
    # a cache larger than every operand tile together: each tile is read once
    M, N, K, tm, tn, tk = 1000, 1200, 300, 128, 256, 64
    gm, gn, gk = math.ceil(M / tm), math.ceil(N / tn), math.ceil(K / tk)
    rc, h, m, b = swz.swz_l2_model_bytes(to.SERPENTINE, 2, M, N, K, tm, tn, tk, 2, 1 << 40, 7, 1,
                                         l2_partitions=2)
    assert rc == 0 and m == gm * gk + gk * gn
    assert b == gm * gk * tm * tk * 2 + gk * gn * tk * tn * 2


def test_native_model_rejects_bad_args(swz):
    assert swz.swz_l2_model(9, 1, 64, 64, 64, 16, 16, 16, 2, 1024, 4, 1)[0] == swz.SWZ_EINVAL
    assert swz.swz_l2_model(to.PANEL, 0, 64, 64, 64, 16, 16, 16, 2, 1024, 4, 1)[0] == swz.SWZ_EINVAL
    assert swz.swz_l2_model(to.ROW, 1, 64, 64, 64, 16, 16, 16, 2, 1024, 0, 1)[0] == swz.SWZ_EINVAL
    assert swz.swz_l2_model_bytes(to.ROW, 1, 64, 64, 64, 16, 16, 16, 2, 1024, 4, 1,
                                  l2_partitions=0)[0] == swz.SWZ_EINVAL
    assert swz.swz_l2_model_bytes(to.ROW, 1, 64, 64, 64, 16, 16, 16, 2, 1024, 4, 1,
                                  k_alternate=2)[0] == swz.SWZ_EINVAL
