"""split_tail: the last wave's tiles are cut into two halves of N width
tile_n/2 when at most half the programs would otherwise be busy.  Results
equal the oracle exactly on integer inputs; the schedule of the other tiles is
unchanged (trace), and each split tile is written by one of its two
half-owners."""
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


CASES = [
    (768, 640, 1024, dict(tile_n=128), 7),    # 30 tiles, P = 7: R = 2 -> 4 halves
    (1000, 1000, 520, dict(tile_n=256), 5),   # 32 tiles of 128 x 256, R = 2 -> 4 halves of 128
    (768, 640, 192, dict(cta_pair=True), 8),  # 9 cluster tiles, 4 clusters: R = 1
    (1280, 1024, 576, dict(cta_pair=True), 10),  # 20 cluster tiles, 5 clusters: R = 0 (no split)
]


@pytest.mark.parametrize("M,N,K,cfg,programs", CASES)
@pytest.mark.parametrize("order,g", [("panel", 2), ("serpentine", 3), ("row", 1)])
def test_split_tail_exact(swz, M, N, K, cfg, programs, order, g):
    A, B = si.small_int_gemm_inputs(M, N, K, "fp16", lo=-4, hi=4, seed=K + programs)
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, num_programs=programs, split_tail=True,
                 **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


def test_split_tail_trace(swz):
    # 6 x 5 grid of 128 x 128 tiles, 7 programs: ids 0..27 are whole tiles on
    # program id mod 7; the tail ids 28, 29 are split between programs 0/1 and 2/3
    A, B = si.gemm_inputs(768, 640, 128, "fp16", "uniform", seed=1)
    trace = torch.full((30 * 2,), -1, dtype=torch.int32, device="cuda")
    C = swz.gemm(A.cuda(), B.cuda(), "panel", 4, True, tile_n=128, num_programs=7, trace=trace,
                 split_tail=True)
    swz.check_status()
    got = trace.view(6, 5, 2).cpu().tolist()
    seq = to.tile_sequence(to.PANEL, 6, 5, 4)
    for pid, (m, n) in enumerate(seq):
        prog, it = got[m][n]
        if pid < 28:
            assert (prog, it) == (pid % 7, pid // 7)
        else:
            j = pid - 28
            assert prog in (2 * j, 2 * j + 1)
            assert it == 4  # after the four whole tiles of programs 0..3
    mx, rel = errors(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())
    assert mx <= MAX_ABS and rel <= REL_FRO


@pytest.mark.parametrize("cfg", [dict(cta_pair=True), dict(tile_n=256)])
def test_split_tail_4096(swz, cfg):
    A, B = si.gemm_inputs(4096, 4096, 4096, "fp16", "uniform", seed=3)
    Ad, Bd = A.cuda(), B.cuda()
    C = swz.gemm(Ad, Bd, "panel", 8, True, split_tail=True, **cfg)
    swz.check_status()
    ii, jj = si.sample_indices(4096, 4096, 128, 128, 1, seed=4)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    mx, rel = errors(got, ref.gemm_entries_f64(A, B, ii, jj))
    assert mx <= MAX_ABS and rel <= REL_FRO
    # identical summation order per element: bitwise equal to whole tiles
    assert torch.equal(C, swz.gemm(Ad, Bd, "panel", 8, True, **cfg))


def test_split_tail_errors(swz):
    A = torch.zeros((768, 128), dtype=torch.float16, device="cuda")
    B = torch.zeros((128, 640), dtype=torch.float16, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.gemm(A, B, "row", 1, False, tile_n=128, split_tail=True)
    assert e.value.code == swz.SWZ_EINVAL
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.gemm(A, B, "row", 1, True, tile_n=128, num_programs=7, split_tail=True,
                 stream_k=True, workspace=ws)
    assert e.value.code == swz.SWZ_EINVAL
