"""CTA pair with 128-wide tiles (cta_pair, tile_n=128): cluster tiles 256 x 128,
tcgen05 cta_group::2 MMAs of 256 x 128, CTA tiles 128 x 128 -- the tile grid
of the 128 x 128 configurations with half the B bytes per CTA.

Exact on small-integer inputs in every mode it shares with the other tile
shapes (persistent or not, both B layouts, TF32, Stream-K, split tail with
B as N x K, dynamic scheduler, 64- and 32-byte spans); the per-tile trace
equals the oracle's persistent schedule on the 256 x 128 cluster grid; the
6144 x 10240 x 4096 configuration meets the tolerance on sampled outputs.
"""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref
from oracle import tile_order as to

pytestmark = pytest.mark.gpu

P128 = dict(cta_pair=True, tile_n=128)


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


@pytest.mark.parametrize("shape", [(300, 392, 200), (256, 128, 64), (1, 8, 8), (129, 136, 72),
                                   (513, 264, 1000), (768, 640, 576)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("b_t", [False, True])
def test_exact_integer(swz, shape, dtype, b_t):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-4, hi=4, seed=M + N + K)
    want = ref.gemm_f64(A, B)
    Bd = B.t().contiguous().cuda() if b_t else B.cuda()
    for persistent in (False, True):
        for order, g in ((to.PANEL, 4), (to.SERPENTINE, 2)):
            C = swz.gemm(A.cuda(), Bd, order, g, persistent, b_transposed=b_t, **P128)
            swz.check_status()
            assert torch.equal(C.cpu().double(), want), (shape, persistent, order)


def test_tf32_exact(swz):
    M, N, K = 513, 264, 100
    g = torch.Generator().manual_seed(9)
    A = torch.randint(-8, 9, (M, K), generator=g).float()
    B = torch.randint(-8, 9, (K, N), generator=g).float()
    C = swz.gemm(A.cuda(), B.cuda(), "panel", 4, True, **P128)  # B transposed inside
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("programs", [6, 8])
def test_tails_and_modes(swz, programs):
    M, N, K = 768, 640, 576
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=programs)
    want = ref.gemm_f64(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    # Stream-K
    n = swz.workspace_size(M, N, K, True, num_programs=programs, **P128)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C = swz.gemm(Ad, Bd, "panel", 2, True, num_programs=programs, stream_k=True, workspace=ws,
                 **P128)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)
    # dynamic scheduler
    C = swz.gemm(Ad, Bd, "serpentine", 2, True, num_programs=programs, dynamic=True,
                 workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"), **P128)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)
    # swizzle spans
    for span in (64, 32):
        C = swz.gemm(Ad, Bd, "row", 1, True, num_programs=programs, smem_swizzle=span, **P128)
        swz.check_status()
        assert torch.equal(C.cpu().double(), want), span


@pytest.mark.parametrize("order,g", [(to.PANEL, 2), (to.SERPENTINE, 2), (to.ROW, 1)])
@pytest.mark.parametrize("programs", [0, 8, 4])
def test_trace(swz, order, g, programs):
    # 768 x 640 with 256 x 128 cluster tiles: a 3 x 5 cluster grid, 6 x 5 CTA tiles
    A, B = si.gemm_inputs(768, 640, 192, "fp16", "uniform", seed=2)
    trace = torch.full((6 * 5 * 2,), -1, dtype=torch.int32, device="cuda")
    persistent = programs > 0
    C = swz.gemm(A.cuda(), B.cuda(), order, g, persistent, num_programs=programs, trace=trace,
                 **P128)
    swz.check_status()
    want = to.persistent_trace(order, 6, 5, g, programs if persistent else 30, cluster_m=2)
    got = trace.view(6, 5, 2).cpu().tolist()
    assert {(m, n): tuple(got[m][n]) for m in range(6) for n in range(5)} == want
    mx, rel = errors(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())
    assert mx <= MAX_ABS and rel <= REL_FRO


@pytest.mark.parametrize("order,g", [(to.ROW, 1), (to.PANEL, 8), (to.SERPENTINE, 8)])
def test_cfg4_sampled(swz, order, g):
    M, N, K = 6144, 10240, 4096
    A, B = si.gemm_inputs(M, N, K, "fp16", "uniform", seed=0)
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, **P128)
    swz.check_status()
    ii, jj = si.sample_indices(M, N, 128, 128, 2, seed=11)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().double().numpy()
    assert np.abs(got - want).max() <= MAX_ABS
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= REL_FRO
