"""swz_gemm_host_tiled (host buffers, C in blocks finished in a growing
square, pitched copies of B panels and C blocks) gives the oracle's result:
exactly on integer inputs for every block count, ragged M / N, both B
layouts and TF32; bit-identical to the row-slab pipeline on real inputs at
8192^3; degenerate shapes and bad arguments handled on the host."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _run(swz, A, B, blocks, **kw):
    M, K = A.shape
    N = B.shape[0] if (kw.get("b_transposed") or A.dtype == torch.float32) else B.shape[1]
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    dA = torch.empty_like(A, device="cuda")
    dB = torch.empty_like(B, device="cuda")
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    swz.gemm_host(hA, hB, hC, dA, dB, dC, blocks=blocks, **kw)
    torch.cuda.current_stream().synchronize()
    swz.check_status()
    return hC


@pytest.mark.parametrize("M,N,K", [(1000, 392, 200), (256, 256, 64), (1, 8, 8), (2048, 1640, 520),
                                   (600, 3000, 64)])
@pytest.mark.parametrize("blocks", [0, 1, 2, 3, 8])
@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(cta_pair=True)])
def test_tiled_exact(swz, M, N, K, blocks, cfg):
    A, B = si.small_int_gemm_inputs(M, N, K, "fp16", lo=-4, hi=4, seed=M + N + blocks)
    C = _run(swz, A, B, blocks, order="serpentine", group=2, **cfg)
    assert torch.equal(C.double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("blocks", [2, 4])
def test_tiled_b_transposed_and_tf32(swz, blocks):
    M, N, K = 1100, 1304, 136
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-4, hi=4, seed=blocks)
    C = _run(swz, A, B.t().contiguous(), blocks, order="panel", group=4, cta_pair=True,
             b_transposed=True)
    assert torch.equal(C.double(), ref.gemm_f64(A, B))
    g = torch.Generator().manual_seed(blocks)
    A32 = torch.randint(-8, 9, (M, K), generator=g).float()
    B32 = torch.randint(-8, 9, (K, N), generator=g).float()
    C = _run(swz, A32, B32.t().contiguous(), blocks, order="panel", group=4, cta_pair=True)
    assert torch.equal(C.double(), ref.gemm_f64(A32, B32))


def test_tiled_8192_equals_slabs(swz):
    A, B = si.gemm_inputs(8192, 8192, 8192, "bf16", "normal", seed=0)
    C = _run(swz, A, B, 4, order="serpentine", group=8, cta_pair=True)
    ii, jj = si.sample_indices(8192, 8192, 128, 256, 1, seed=5)
    mx, rel = errors(C.numpy()[ii, jj], ref.gemm_entries_f64(A, B, ii, jj))
    assert mx <= MAX_ABS and rel <= REL_FRO
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty((8192, 8192), dtype=torch.float32).pin_memory()
    dA, dB = torch.empty_like(A, device="cuda"), torch.empty_like(B, device="cuda")
    dC = torch.empty((8192, 8192), dtype=torch.float32, device="cuda")
    swz.gemm_host(hA, hB, hC, dA, dB, dC, "serpentine", 8, slabs=8, cta_pair=True)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(C, hC)


def test_tiled_degenerate_and_errors(swz):
    A = torch.zeros((64, 0), dtype=torch.float16)
    B = torch.zeros((0, 32), dtype=torch.float16)
    C = _run(swz, A, B, 2, order="row", group=1, tile_n=128)
    assert torch.count_nonzero(C).item() == 0
    s = torch.cuda.current_stream().cuda_stream
    o = swz.make_opts()
    d = torch.empty(1024, dtype=torch.float32, device="cuda")
    h = torch.empty(1024, dtype=torch.float32).pin_memory()
    args = (h.data_ptr(), h.data_ptr(), h.data_ptr(), 16, 16, 16, 0, 1, o, d.data_ptr(),
            d.data_ptr(), d.data_ptr())
    assert swz.swz_gemm_host_tiled(*args, 9, s) == swz.SWZ_EINVAL       # more than 8 blocks
    assert swz.swz_gemm_host_tiled(*args, -1, s) == swz.SWZ_EINVAL
    bad = (h.data_ptr(), h.data_ptr(), h.data_ptr(), 16, 12, 16, 0, 1, o, d.data_ptr(),
           d.data_ptr(), d.data_ptr())
    assert swz.swz_gemm_host_tiled(*bad, 2, s) == swz.SWZ_EINVAL        # N % 8 for K x N B
