"""Stream-K tail (swz_gemm_opts.stream_k): the last partial wave of tiles is
split along K among all programs; results must equal the oracle exactly on
integer inputs, within tolerance on real inputs, and be bit-identical from run
to run (the pieces of a tile are always added in K order)."""
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


def _ws(swz, M, N, K, **kw):
    n = swz.workspace_size(M, N, K, True, **kw)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda"), n


# (M, N, K, cfg, programs): programs chosen so that tiles % clusters != 0;
# K values give tail ranges longer and shorter than one cluster (the latter
# leaves some programs with an empty range).  kb = K blocks of a tile: one
# stage each, 64 elements of K (128 for 128-wide tiles, two-atom stages).
CASES = [
    (768, 640, 1024, dict(tile_n=128), 7),       # 30 tiles, R = 2, kb = 8
    (768, 640, 192, dict(tile_n=128), 7),        # kb = 2: I = 4 < 7 programs
    (768, 640, 64, dict(tile_n=128), 7),         # kb = 1: no split possible
    (1000, 1000, 520, dict(tile_n=256), 5),      # ragged M/N/K
    (768, 640, 1024, dict(cta_pair=True), 4),    # 9 cluster tiles, 2 clusters, R = 1
    (1280, 1024, 576, dict(cta_pair=True), 6),   # 20 cluster tiles, 3 clusters
    (768, 640, 192, dict(cta_pair=True), 8),     # kb = 3, 4 clusters, R = 1: I = 3 < 4
    # a few tiles over every resident program (0): more reducers per tile
    # than chunks per warp row, the fine reduction; ragged M and N
    (200, 360, 8192, dict(cta_pair=True), 0),    # 2 cluster tiles, ~38 clusters each
    (100, 256, 4096, dict(tile_n=256), 0),       # 1 tile, 64 K blocks over 64 programs
    (300, 200, 8192, dict(tile_n=128), 0),       # 6 tiles of 128 x 128, ~25 programs each
]


@pytest.mark.parametrize("M,N,K,cfg,programs", CASES)
@pytest.mark.parametrize("order,g", [("panel", 2), ("serpentine", 3), ("row", 1)])
def test_stream_k_integer_exact(swz, M, N, K, cfg, programs, order, g):
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=K + programs)
    ws, n = _ws(swz, M, N, K, num_programs=programs, **cfg)
    assert n > 0 or K == 0
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, num_programs=programs, stream_k=True,
                 workspace=ws, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("cfg", [dict(tile_n=256), dict(cta_pair=True)])
def test_stream_k_4096_fp16(swz, cfg):
    A, B = si.gemm_inputs(4096, 4096, 4096, "fp16", "uniform", seed=5)
    ws, n = _ws(swz, 4096, 4096, 4096, **cfg)
    assert n > 0  # 512 (256) tiles do not divide evenly over the resident programs
    Ad, Bd = A.cuda(), B.cuda()
    C1 = swz.gemm(Ad, Bd, "panel", 8, True, stream_k=True, workspace=ws, **cfg)
    C2 = swz.gemm(Ad, Bd, "panel", 8, True, stream_k=True, workspace=ws, **cfg)
    swz.check_status()
    assert torch.equal(C1, C2)  # deterministic
    ii, jj = si.sample_indices(4096, 4096, 128, 256, 2, seed=9)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C1[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    mx, rel = errors(got, want)
    assert mx <= MAX_ABS and rel <= REL_FRO
    # and it agrees with the whole-tile schedule to FP32 summation order
    C0 = swz.gemm(Ad, Bd, "panel", 8, True, **cfg)
    assert (C0 - C1).abs().max().item() <= 1e-3


def test_stream_k_8192_bf16_pair(swz):
    A, B = si.gemm_inputs(8192, 8192, 8192, "bf16", "normal", seed=0)
    ws, n = _ws(swz, 8192, 8192, 8192, cta_pair=True)
    C = swz.gemm(A.cuda(), B.cuda(), "panel", 8, True, cta_pair=True, stream_k=True, workspace=ws)
    swz.check_status()
    ii, jj = si.sample_indices(8192, 8192, 128, 256, 1, seed=3)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    mx, rel = errors(got, want)
    assert mx <= MAX_ABS and rel <= REL_FRO
    assert torch.isfinite(C).all().item()


def test_stream_k_errors(swz):
    A = torch.zeros((768, 128), dtype=torch.float16, device="cuda")
    B = torch.zeros((128, 640), dtype=torch.float16, device="cuda")
    ws, n = _ws(swz, 768, 640, 128, tile_n=128, num_programs=7)
    with pytest.raises(swz.SwzError) as e:  # not persistent
        swz.gemm(A, B, "row", 1, False, tile_n=128, stream_k=True, workspace=ws)
    assert e.value.code == swz.SWZ_EINVAL
    with pytest.raises(swz.SwzError) as e:  # workspace too small
        swz.gemm(A, B, "row", 1, True, tile_n=128, num_programs=7, stream_k=True,
                 workspace=ws[: n // 2])
    assert e.value.code == swz.SWZ_EINVAL
    with pytest.raises(swz.SwzError) as e:  # no workspace
        swz.gemm(A, B, "row", 1, True, tile_n=128, num_programs=7, stream_k=True)
    assert e.value.code == swz.SWZ_EINVAL
    big = torch.zeros((8192, 128), dtype=torch.float16, device="cuda")
    B2 = torch.zeros((128, 8192), dtype=torch.float16, device="cuda")
    with pytest.raises(swz.SwzError) as e:  # more programs than can be resident
        swz.gemm(big, B2, "row", 1, True, tile_n=128, num_programs=4000, stream_k=True,
                 workspace=ws)
    assert e.value.code == swz.SWZ_EUNSUPPORTED
    # evenly divisible tiles need no workspace and run whole tiles
    assert swz.workspace_size(768, 640, 128, True, tile_n=128, num_programs=6) == 0


# (M, N, K, cfg, programs): whole units and a tail; more programs than tiles
# (every tile split); CTA pairs with a tail; one cluster tile over 8 clusters
TRACE_CASES = [
    (768, 640, 1024, dict(tile_n=128), 7),
    (768, 640, 384, dict(tile_n=128), 40),
    (768, 640, 192, dict(tile_n=256), 5),
    (1280, 1024, 576, dict(cta_pair=True), 6),
    (256, 256, 4096, dict(cta_pair=True), 16),
]


@pytest.mark.parametrize("M,N,K,cfg,programs", TRACE_CASES)
@pytest.mark.parametrize("order,g", [(to.PANEL, 2), (to.SERPENTINE, 3)])
def test_stream_k_trace_matches_oracle(swz, M, N, K, cfg, programs, order, g):
    # which program writes each tile, at which item of its loop: the
    # schedule the oracle writes out from the Stream-K definition
    rc, (tm, tn, _, _, P) = swz.swz_gemm_plan(
        M, N, K, 1, swz.make_opts(stream_k=True, num_programs=programs, **cfg))
    assert rc == swz.SWZ_OK and P == programs
    kb = -(-K // (128 if cfg.get("tile_n") == 128 else 64))  # K blocks per stage
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=K + programs)
    ws, n = _ws(swz, M, N, K, num_programs=programs, **cfg)
    trace = torch.full((tm * tn * 2,), -1, dtype=torch.int32, device="cuda")
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, num_programs=programs, stream_k=True,
                 workspace=ws, trace=trace, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))
    want = to.stream_k_trace(order, tm, tn, g, P, kb, cluster_m=2 if cfg.get("cta_pair") else 1)
    got = trace.view(tm, tn, 2).cpu().tolist()
    assert {(m, n): tuple(got[m][n]) for m in range(tm) for n in range(tn)} == want
