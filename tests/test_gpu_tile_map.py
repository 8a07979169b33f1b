"""Device tile maps (swz_tile_map) are bit-identical to the oracle's."""
import random

import pytest

from gpu_util import require_gpu
from oracle import tile_order as to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


CASES = [(o, 8, 8, g) for o, g in [(to.ROW, 1), (to.COL, 1), (to.PANEL, 4), (to.MORTON, 1),
                                    (to.XOR, 1), (to.SERPENTINE, 2)]]
CASES += [(to.PANEL, 4, 4, 2), (to.SERPENTINE, 4, 4, 2)]
CASES += [(o, 32, 16, g) for o in range(6) for g in (2, 4, 8, 16)]
CASES += [(o, 48, 80, g) for o in range(6) for g in (3, 8, 16)]
CASES += [(o, 3, 5, 2) for o in range(6)] + [(o, 1, 1, 1) for o in range(6)]


@pytest.mark.parametrize("order,gm,gn,g", CASES)
def test_tile_map_bit_exact(swz, order, gm, gn, g):
    m, n = swz.tile_map(order, gm, gn, g)
    assert list(zip(m.tolist(), n.tolist())) == to.tile_sequence(order, gm, gn, g)


def test_tile_map_random_grids(swz):
    rnd = random.Random(7)
    for _ in range(40):
        order = rnd.randrange(6)
        gm, gn, g = rnd.randint(1, 90), rnd.randint(1, 90), rnd.randint(1, 20)
        m, n = swz.tile_map(order, gm, gn, g)
        assert list(zip(m.tolist(), n.tolist())) == to.tile_sequence(order, gm, gn, g), (order, gm, gn, g)


def test_tile_map_large_grid(swz):
    # 64 x 64 cluster tiles = the 8192^3 2-CTA grid at 128-row CTA tiles
    for order, g in [(to.PANEL, 16), (to.SERPENTINE, 8), (to.MORTON, 1), (to.XOR, 1)]:
        m, n = swz.tile_map(order, 64, 64, g)
        assert list(zip(m.tolist(), n.tolist())) == to.tile_sequence(order, 64, 64, g)
