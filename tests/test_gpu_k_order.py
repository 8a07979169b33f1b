"""The K order of a tile.  A launch with one CTA (or cluster) per tile sums
every tile's K blocks in ascending order; a persistent launch with P programs
(clusters) takes them in descending order for the tiles of odd waves (tile
id / P odd).  On real-valued inputs the two orders round differently, so the
tiles of even waves must equal the one-CTA-per-tile result bit for bit and the
tiles of odd waves must differ from it (with K = 2048, N(0, 1) products, some
element of a 128 x 256 tile differs with overwhelming probability); both stay
within the GEMM tolerance of the oracle.  On integer inputs every order is
exact, including a ragged K, where a descending tile starts on the partial
K block."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref
from oracle import tile_order as to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


@pytest.mark.parametrize("cfg,programs,order,g", [
    (dict(tile_n=256), 6, "row", 1),
    (dict(tile_n=128), 10, "serpentine", 2),
    (dict(cta_pair=True), 6, "panel", 2),
])
def test_tiles_of_odd_waves_run_k_descending(swz, cfg, programs, order, g):
    M, N, K = 1024, 1024, 2048
    A, B = si.gemm_inputs(M, N, K, "bf16", "normal", seed=9)
    Ad, Bd = A.cuda(), B.cuda()
    rc, (tm, tn, sm, sn, P) = swz.swz_gemm_plan(M, N, K, 1, swz.make_opts(num_programs=programs,
                                                                          **cfg))
    assert rc == swz.SWZ_OK and P == programs
    cl = 2 if cfg.get("cta_pair") else 1
    up = swz.gemm(Ad, Bd, order, g, False, **cfg)  # one CTA (cluster) per tile
    C = swz.gemm(Ad, Bd, order, g, True, num_programs=programs, **cfg)
    swz.check_status()
    bm, bn = 128, N // tn
    seen_odd = 0
    omap = {"row": to.ROW, "serpentine": to.SERPENTINE, "panel": to.PANEL}[order]
    for w in range(sm * sn):  # scheduler units: cluster tiles of cl CTA tiles
        um, un = to.tile_of(omap, w, sm, sn, g)
        odd = (w // (P // cl)) % 2 == 1
        for r in range(cl):
            rows = slice((um * cl + r) * bm, (um * cl + r + 1) * bm)
            cols = slice(un * bn, (un + 1) * bn)
            same = torch.equal(C[rows, cols], up[rows, cols])
            assert same != odd, (w, r, odd)
        seen_odd += odd
    assert seen_odd > 0
    ii, jj = si.sample_indices(M, N, 128, 256, 2, seed=3)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    for X in (C, up):
        got = X[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
        mx, rel = errors(got, want)
        assert mx <= MAX_ABS and rel <= REL_FRO


@pytest.mark.parametrize("cfg,programs", [(dict(tile_n=128), 7), (dict(tile_n=256), 5),
                                          (dict(cta_pair=True), 6)])
@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
def test_ragged_k_descending_exact(swz, cfg, programs, dtype):
    # K = 1000 is no multiple of the K block: a tile of an odd wave starts on
    # the partial block, zero-filled past K by TMA; with few programs there
    # are several waves, and integer inputs make every sum exact
    M, N, K = 768, 640, 1000
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=programs)
    want = ref.gemm_f64(A, B)
    if dtype == "tf32":
        A, B = A.float(), B.float()
    C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 2, True, num_programs=programs, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)
