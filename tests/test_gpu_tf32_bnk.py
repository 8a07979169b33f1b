"""B stored transposed (N x K, K-major operand) and the TF32 path (fp32
inputs, the first page's --dtype fp32).

* fp16/bf16 with B as N x K: exact on integer inputs for every tile shape,
  the CTA pair, split tails (half-width boxes) and Stream-K.
* TF32: exact on small-integer inputs (exactly representable in TF32, exact
  fp32 sums); on U[-1, 1) inputs every element must lie within the error
  bound TF32 rounding allows: each operand keeps 10 fraction bits (relative
  error below 2^-10 however it is rounded), so each product is within
  2^-9 + 2^-20 of its exact value relative to |a||b|, and fp32 accumulation
  of K terms adds at most K * 2^-24 relative to sum |a||b|:
      |C - Cref|_ij <= (2^-9 + 2^-20 + K * 2^-24) * (|A| |B|)_ij.
"""
import numpy as np
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


@pytest.mark.parametrize("shape", [(300, 392, 200), (129, 136, 72), (513, 264, 1000), (1, 8, 8)])
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_b_transposed_exact(swz, shape, cfg, dtype):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-4, hi=4, seed=M + N)
    Bt = B.t().contiguous().cuda()
    want = ref.gemm_f64(A, B)
    for persistent in (False, True):
        C = swz.gemm(A.cuda(), Bt, "serpentine", 2, persistent, b_transposed=True, **cfg)
        swz.check_status()
        assert torch.equal(C.cpu().double(), want), (shape, cfg, persistent)


@pytest.mark.parametrize("cfg,programs", [(dict(tile_n=128), 7), (dict(cta_pair=True), 8),
                                          (dict(tile_n=256), 5)])
def test_b_transposed_tails(swz, cfg, programs):
    M, N, K = 768, 640, 576
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=programs)
    Bt = B.t().contiguous().cuda()
    want = ref.gemm_f64(A, B)
    C = swz.gemm(A.cuda(), Bt, "panel", 2, True, num_programs=programs, b_transposed=True, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)
    n = swz.workspace_size(M, N, K, True, num_programs=programs, **cfg)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C = swz.gemm(A.cuda(), Bt, "panel", 2, True, num_programs=programs, stream_k=True,
                 workspace=ws, b_transposed=True, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), want)


def _int_fp32(M, N, K, seed, lo=-8, hi=8):
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(lo, hi + 1, (M, K), generator=g).float()
    B = torch.randint(lo, hi + 1, (K, N), generator=g).float()
    return A, B


@pytest.mark.parametrize("shape", [(256, 256, 64), (300, 392, 36), (129, 136, 100), (513, 264, 1000),
                                   (1, 4, 4)])
@pytest.mark.parametrize("cfg", CFGS)
def test_tf32_integer_exact(swz, shape, cfg):
    M, N, K = shape
    A, B = _int_fp32(M, N, K, seed=M + K)
    want = ref.gemm_f64(A, B)
    for persistent in (False, True):
        C = swz.gemm(A.cuda(), B.cuda(), "panel", 4, persistent, **cfg)  # B transposed inside
        swz.check_status()
        assert torch.equal(C.cpu().double(), want), (shape, cfg, persistent)


def _bound(A, B, K):
    absab = ref.gemm_f64(A.abs(), B.abs()).numpy()
    return (2.0 ** -9 + 2.0 ** -20 + K * 2.0 ** -24) * absab


@pytest.mark.parametrize("cfg", CFGS)
def test_tf32_uniform_within_bound(swz, cfg):
    M, N, K = 1024, 1024, 512
    g = torch.Generator().manual_seed(7)
    A = torch.rand((M, K), generator=g) * 2 - 1
    B = torch.rand((K, N), generator=g) * 2 - 1
    want = ref.gemm_f64(A, B).numpy()
    C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 8, True, **cfg).cpu().double().numpy()
    err = np.abs(C - want)
    assert (err <= _bound(A, B, K)).all(), float((err / _bound(A, B, K)).max())
    assert np.linalg.norm(C - want) / np.linalg.norm(want) <= 2.0 ** -9


def test_tf32_4096_sampled(swz):
    M = N = K = 4096
    g = torch.Generator().manual_seed(8)
    A = torch.rand((M, K), generator=g) * 2 - 1
    B = torch.rand((K, N), generator=g) * 2 - 1
    C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 8, True, cta_pair=True)
    ii, jj = si.sample_indices(M, N, 128, 256, 2, seed=3)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    bound = (2.0 ** -9 + 2.0 ** -20 + K * 2.0 ** -24) * ref.gemm_entries_f64(A.abs(), B.abs(), ii, jj)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().double().numpy()
    assert (np.abs(got - want) <= bound).all()


def test_tf32_wrapper_equals_direct_nk(swz):
    A, B = _int_fp32(512, 384, 256, seed=1, lo=-100, hi=100)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = swz.gemm(Ad, Bd, "row", 1, True, cta_pair=True)
    C2 = swz.gemm(Ad, Bd.t().contiguous(), "row", 1, True, cta_pair=True, b_transposed=True)
    assert torch.equal(C1, C2)


def test_tf32_errors(swz):
    A = torch.zeros((128, 64), dtype=torch.float32, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.float32, device="cuda")
    C = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    opts = swz.make_opts(swz.SWZ_TF32)                       # B as K x N: not taken for TF32
    assert swz.swz_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 128, 64, swz.SWZ_ROW,
                           1, 0, opts, s) == swz.SWZ_EUNSUPPORTED
    opts = swz.make_opts(swz.SWZ_TF32, b_layout=swz.SWZ_B_NK)  # K % 4 != 0
    assert swz.swz_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 128, 62, swz.SWZ_ROW,
                           1, 0, opts, s) == swz.SWZ_EINVAL
