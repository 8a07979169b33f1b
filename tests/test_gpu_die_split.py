"""Die split (swz_gemm_opts.die_split): after swz_calibrate, the clusters on
each die of the package take their own share of the tile order.  Results
must equal the oracle exactly on integer inputs, the plain schedule bit for
bit when tiles are whole, and the per-tile trace must equal the oracle's
die-split schedule for the cluster dies the library reports."""
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


def test_die_split_needs_calibration_first(swz):
    # runs before any calibration in this process (the first test of the
    # only file that calibrates)
    A = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.gemm(A, B, "row", 1, True, die_split=True)
    assert e.value.code == swz.SWZ_EUNSUPPORTED
    rc, _, _, _ = swz.swz_gemm_die_plan(256, 256, 64, swz.make_opts())
    assert rc == swz.SWZ_EUNSUPPORTED


@pytest.fixture(scope="module")
def dies(swz):
    return swz.calibrate()


def test_calibration_finds_two_dies(swz, dies):
    rc, (sms, _, _, _) = swz.swz_device_info()
    assert rc == swz.SWZ_OK and len(dies) == sms
    # a GB300 is two dies; each holds a large share of the SMs
    n1 = sum(dies)
    assert 0.3 * sms < n1 < 0.7 * sms, dies


def _cluster_dies(swz, M, N, K, **cfg):
    rc, info, P0, U0 = swz.swz_gemm_die_plan(M, N, K, swz.make_opts(**cfg))
    assert rc == swz.SWZ_OK
    d = [i >> 15 for i in info]
    # ranks are dense per die and in cluster order
    for die in (0, 1):
        assert [i & 0x7FFF for i in info if i >> 15 == die] == list(range(d.count(die)))
    assert P0 == d.count(0)
    return d, U0


# shapes with at least as many scheduler units as the resident capacity, so
# that the launch is the calibrated full-capacity shape
CASES = [
    (2048, 2048, 256, dict(tile_n=128)),                 # 256 tiles, 1-CTA
    (2560, 2560, 192, dict(cta_pair=True)),              # 100 cluster tiles, pairs
    (2304, 2560, 320, dict(cta_pair=True, tile_n=128)),  # 180 cluster tiles of 256 x 128
]


@pytest.mark.parametrize("M,N,K,cfg", CASES)
@pytest.mark.parametrize("stream_k", [False, True])
def test_die_split_exact_and_trace(swz, dies, M, N, K, cfg, stream_k):
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=M + K)
    Ad, Bd = A.cuda(), B.cuda()
    rc, (tm, tn, _, _, P) = swz.swz_gemm_plan(M, N, K, 1, swz.make_opts(stream_k=stream_k, **cfg))
    assert rc == swz.SWZ_OK
    ws = None
    if stream_k:
        n = swz.workspace_size(M, N, K, True, **cfg)
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    trace = torch.full((tm * tn * 2,), -1, dtype=torch.int32, device="cuda")
    C = swz.gemm(Ad, Bd, "serpentine", 3, True, die_split=True, trace=trace, stream_k=stream_k,
                 workspace=ws, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))
    if not stream_k:  # whole tiles: the plain schedule, bit for bit
        C0 = swz.gemm(Ad, Bd, "serpentine", 3, True, **cfg)
        assert torch.equal(C, C0)
    d, _ = _cluster_dies(swz, M, N, K, **cfg)
    cm = 2 if cfg.get("cta_pair") else 1
    assert len(d) * cm == P
    kb = -(-K // (128 if cfg.get("tile_n") == 128 else 64)) if stream_k else None
    want = to.die_split_trace(to.SERPENTINE, tm, tn, 3, d, k_blocks=kb, cluster_m=cm)
    got = trace.view(tm, tn, 2).cpu().tolist()
    assert {(m, n): tuple(got[m][n]) for m in range(tm) for n in range(tn)} == want


def test_die_split_8192_bf16_pair(swz, dies):
    A, B = si.gemm_inputs(8192, 8192, 8192, "bf16", "normal", seed=4)
    Ad, Bd = A.cuda(), B.cuda()
    # whole tiles: every tile's K loop is the plain schedule's, bit for bit
    C1 = swz.gemm(Ad, Bd, "serpentine", 8, True, cta_pair=True, die_split=True)
    C0 = swz.gemm(Ad, Bd, "serpentine", 8, True, cta_pair=True)
    swz.check_status()
    assert torch.equal(C0, C1)
    # with Stream-K each die splits its own tail, so other tiles are split at
    # other K blocks: within the GEMM tolerance of the oracle, deterministic
    n = swz.workspace_size(8192, 8192, 8192, True, cta_pair=True)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    C2 = swz.gemm(Ad, Bd, "serpentine", 8, True, cta_pair=True, die_split=True, stream_k=True,
                  workspace=ws)
    C3 = swz.gemm(Ad, Bd, "serpentine", 8, True, cta_pair=True, die_split=True, stream_k=True,
                  workspace=ws)
    swz.check_status()
    assert torch.equal(C2, C3)
    ii, jj = si.sample_indices(8192, 8192, 128, 256, 1, seed=6)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C2[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    mx, rel = errors(got, want)
    assert mx <= MAX_ABS and rel <= REL_FRO


def test_die_split_other_launches_run_the_plain_schedule(swz, dies):
    # fewer tiles than the capacity: the launch is not the calibrated shape
    A, B = si.small_int_gemm_inputs(512, 512, 128, "fp16", lo=-3, hi=3, seed=5)
    trace = torch.full((4 * 2 * 2,), -1, dtype=torch.int32, device="cuda")
    C = swz.gemm(A.cuda(), B.cuda(), "row", 1, True, tile_n=256, die_split=True, trace=trace)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))
    assert {(m, n): tuple(trace.view(4, 2, 2).cpu().tolist()[m][n]) for m in range(4)
            for n in range(2)} == to.persistent_trace(to.ROW, 4, 2, 1, 8)
    with pytest.raises(swz.SwzError) as e:  # not with the dynamic scheduler
        swz.gemm(A.cuda(), B.cuda(), "row", 1, True, die_split=True, dynamic=True,
                 workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"))
    assert e.value.code == swz.SWZ_EINVAL
    with pytest.raises(swz.SwzError) as e:  # persistent launches only
        swz.gemm(A.cuda(), B.cuda(), "row", 1, False, die_split=True)
    assert e.value.code == swz.SWZ_EINVAL
