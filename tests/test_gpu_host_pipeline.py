"""swz_gemm_host (host buffers in and out, copies overlapped with the GEMM in
row slabs) gives the oracle's result: exactly on integer inputs, within
tolerance at 8192^3, for every slab count, ragged M, and the degenerate
shapes."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _run(swz, A, B, slabs, **kw):
    M, K = A.shape
    N = B.shape[1]
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(A, device="cuda")
    dB = torch.empty_like(B, device="cuda")
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    swz.gemm_host(hA, hB, hC, dA, dB, dC, slabs=slabs, **kw)
    torch.cuda.current_stream().synchronize()
    swz.check_status()
    return hC


@pytest.mark.parametrize("M,N,K", [(1000, 392, 200), (256, 256, 64), (1, 8, 8), (2048, 640, 520)])
@pytest.mark.parametrize("slabs", [1, 2, 3, 64])
@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(cta_pair=True)])
def test_host_pipeline_exact(swz, M, N, K, slabs, cfg):
    A, B = si.small_int_gemm_inputs(M, N, K, "fp16", lo=-4, hi=4, seed=M + slabs)
    C = _run(swz, A, B, slabs, order="serpentine", group=2, **cfg)
    assert torch.equal(C.double(), ref.gemm_f64(A, B))


def test_host_pipeline_8192(swz):
    A, B = si.gemm_inputs(8192, 8192, 8192, "bf16", "normal", seed=0)
    C = _run(swz, A, B, 4, order="panel", group=8, cta_pair=True)
    ii, jj = si.sample_indices(8192, 8192, 128, 256, 1, seed=5)
    mx, rel = errors(C.numpy()[ii, jj], ref.gemm_entries_f64(A, B, ii, jj))
    assert mx <= MAX_ABS and rel <= REL_FRO
    # against the device-resident call: a slab launch is a launch of its own,
    # whose waves (and so the K direction of each tile) differ, so the two
    # agree within the GEMM tolerance rather than bit for bit
    D = swz.gemm(A.cuda(), B.cuda(), "panel", 8, True, cta_pair=True)
    mx, rel = errors(C.numpy(), D.cpu().numpy())
    assert mx <= MAX_ABS and rel <= REL_FRO


def test_host_pipeline_degenerate(swz):
    A = torch.zeros((64, 0), dtype=torch.float16)
    B = torch.zeros((0, 32), dtype=torch.float16)
    C = _run(swz, A, B, 2, order="row", group=1, tile_n=128)
    assert torch.count_nonzero(C).item() == 0
    hA = torch.zeros((0, 16), dtype=torch.float16)
    hB = torch.zeros((16, 8), dtype=torch.float16)
    rc = swz.swz_gemm_host(hA.data_ptr(), hB.data_ptr(), 0, 0, 8, 16, swz.SWZ_ROW, 1, None,
                           0, 0, 0, 0, 0)
    assert rc == swz.SWZ_OK


def test_host_pipeline_refuses_before_enqueue(swz):
    # Morton on 1536-row slabs of 128 x 128 tiles: a 12 x 8 grid, not a permutation
    A = torch.zeros((3072, 64), dtype=torch.float16)
    B = torch.zeros((64, 1024), dtype=torch.float16)
    with pytest.raises(swz.SwzError) as e:
        _run(swz, A, B, 2, order="morton", group=1, tile_n=128)
    assert e.value.code == swz.SWZ_ENOTBIJECTIVE
