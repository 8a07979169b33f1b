"""Sizes at the edges of the index arithmetic.

- C with more than 2^31 elements (49152 x 49152): element offsets past the
  32-bit range in the epilogue's stores and clipping.
- K = 2^20: 16384 K blocks of 64, so the stage ring's phase bits wrap
  thousands of times in one tile, and with Stream-K a single tile's K range
  is spread over every resident program.
- A transpose of more than 2^31 words (65536 x 40000).

Integer-valued operands in [-3, 3] keep every partial and final sum an
integer of magnitude at most 9 * 2^20 < 2^24, exact in FP32 whatever the
summation order, so the GEMMs are compared with the oracle exactly."""
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


@pytest.mark.parametrize("cfg,persistent", [(dict(cta_pair=True), True),
                                            (dict(tile_n=256), True),
                                            (dict(tile_n=128), False)])
def test_c_beyond_2_31_elements(swz, cfg, persistent):
    M = N = 49152
    K = 64
    assert M * N > 2**31
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=31)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    swz.gemm(A.cuda(), B.cuda(), "panel", 8, persistent, out=C, **cfg)
    swz.check_status()
    assert not torch.isnan(C).any().item()  # every tile written
    # the last 128 rows in full: their offsets are all beyond 2^31 elements
    assert (M - 128) * N > 2**31
    assert torch.equal(C[M - 128:].cpu().double(), ref.gemm_f64(A, B, M - 128, M))
    ii, jj = si.sample_indices(M, N, 1024, 1024, 2, seed=3)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().double().numpy()
    assert np.array_equal(got, want)


@pytest.fixture(scope="module")
def long_k():
    M = N = 256
    K = 1 << 20
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=41)
    ii, jj = si.sample_indices(M, N, 32, 32, 4, seed=5)
    return A, B, ii, jj, ref.gemm_entries_f64(A, B, ii, jj)


@pytest.mark.parametrize("cfg", [dict(cta_pair=True), dict(tile_n=256),
                                 dict(cta_pair=True, stream_k=True),
                                 dict(tile_n=128, stream_k=True)])
def test_k_2_20(swz, long_k, cfg):
    A, B, ii, jj, want = long_k
    M, K = A.shape
    N = B.shape[1]
    ws = None
    if cfg.get("stream_k"):
        n = swz.workspace_size(M, N, K, True, **{k: v for k, v in cfg.items()
                                                  if k != "stream_k"})
        assert n > 0  # fewer tiles than programs: the whole K range is split
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    swz.gemm(A.cuda(), B.cuda(), "serpentine", 2, True, out=C, workspace=ws, **cfg)
    swz.check_status()
    assert not torch.isnan(C).any().item()
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().double().numpy()
    assert np.array_equal(got, want)


@pytest.fixture(scope="module")
def big_words():
    M, N = 65536, 40000
    assert M * N > 2**31
    return si.device_words(M, N, seed=51)


@pytest.mark.parametrize("layout", ["naive", "padded", "xor"])
def test_transpose_beyond_2_31_words(swz, big_words, layout):
    x = big_words
    M, N = x.shape
    y = torch.empty((N, M), dtype=torch.int32, device="cuda")
    swz.transpose(x, layout, out=y)
    torch.cuda.synchronize()
    # 64 x 64 blocks against the oracle, three of them past 2^31 words
    for r0, c0 in ((0, 0), (0, N - 64), (M - 64, 0), (54000, 20000), (M - 64, N - 64)):
        xb = x[r0:r0 + 64, c0:c0 + 64].cpu()
        assert torch.equal(y[c0:c0 + 64, r0:r0 + 64].cpu(), ref.transpose_u32(xb)), (r0, c0)
    # every word: y^T == x, compared on the device in bands of rows of x
    for r0 in range(0, M, 4096):
        assert torch.equal(y[:, r0:r0 + 4096].t(), x[r0:r0 + 4096]), r0
