"""Operand-stage swizzle spans of the tcgen05 GEMM (smem_swizzle 128 / 64 / 32).

The span changes only where the bytes of a stage sit in shared memory (and
how many TMA boxes fill it), never the arithmetic: on small-integer inputs
every mode is exact against the oracle, and on real-valued inputs the modes
agree bit for bit (the tensor core sums the same products in the same order).
Shapes cover the one-box (3-D map) and per-group (2-D boxes) load paths:
K a multiple of the span's element count or not, N a multiple of the B box
width or not, ragged M / N / K edges, half-width tail tiles and Stream-K.
"""
import pytest
import torch

import synth_inputs as si
from gpu_util import require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


CFGS = [dict(tile_n=128), dict(tile_n=256), dict(cta_pair=True)]
SPANS = [32, 64, 128]


@pytest.mark.parametrize("shape", [(256, 512, 512), (300, 392, 200), (129, 136, 72),
                                   (513, 264, 1000), (1, 8, 8)])
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("span", SPANS)
@pytest.mark.parametrize("b_t", [False, True])
def test_exact_integer(swz, shape, cfg, span, b_t):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, "fp16", lo=-4, hi=4, seed=M + K + span)
    want = ref.gemm_f64(A, B)
    Bd = B.t().contiguous().cuda() if b_t else B.cuda()
    for persistent in (False, True):
        C = swz.gemm(A.cuda(), Bd, "serpentine", 2, persistent, b_transposed=b_t,
                     smem_swizzle=span, **cfg)
        swz.check_status()
        assert torch.equal(C.cpu().double(), want), (shape, cfg, span, b_t, persistent)


@pytest.mark.parametrize("span", [32, 64])
@pytest.mark.parametrize("cfg", CFGS)
def test_tf32_exact(swz, span, cfg):
    M, N, K = 300, 264, 100  # K % 8 == 4: the last column group is partial
    g = torch.Generator().manual_seed(span)
    A = torch.randint(-8, 9, (M, K), generator=g).float()
    B = torch.randint(-8, 9, (K, N), generator=g).float()
    C = swz.gemm(A.cuda(), B.t().contiguous().cuda(), "panel", 4, True, b_transposed=True,
                 smem_swizzle=span, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("cfg,programs", [(dict(tile_n=128), 7), (dict(cta_pair=True), 8)])
@pytest.mark.parametrize("span", [32, 64])
def test_tails(swz, cfg, programs, span):
    M, N, K = 768, 640, 576
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=programs + span)
    want = ref.gemm_f64(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    C = swz.gemm(Ad, Bd, "panel", 2, True, num_programs=programs, smem_swizzle=span, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)
    n = swz.workspace_size(M, N, K, True, num_programs=programs, **cfg)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C = swz.gemm(Ad, Bd, "panel", 2, True, num_programs=programs, stream_k=True, workspace=ws,
                 smem_swizzle=span, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)


@pytest.mark.parametrize("cfg", CFGS)
def test_modes_bit_identical(swz, cfg):
    M = N = 1024
    K = 512
    A, B = si.gemm_inputs(M, N, K, "fp16", "uniform", seed=1)
    Ad, Bd = A.cuda(), B.cuda()
    outs = [swz.gemm(Ad, Bd, "panel", 8, True, smem_swizzle=s, **cfg) for s in SPANS]
    swz.check_status()
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[2])


def test_invalid_span(swz):
    A = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.float16, device="cuda")
    C = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for bad in (16, 96, 256, -64):
        opts = swz.make_opts(smem_swizzle=bad)
        assert swz.swz_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 128, 64,
                               swz.SWZ_ROW, 1, 0, opts, s) == swz.SWZ_EINVAL
