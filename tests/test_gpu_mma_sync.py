"""swz_gemm_mma_sync (cp.async / ldmatrix / mma.sync path with a run-time
shared-memory operand layout) equals the oracle exactly on integer inputs
for every layout, and within tolerance on real inputs."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu

LAYOUTS = [(8, 1, 1, 0), (8, 1, 1, 8), (8, 1, 8, 0), (8, 2, 4, 0), (16, 1, 4, 0), (8, 4, 2, 16),
           (8, 1, 8, 8)]


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", [(256, 256, 128), (300, 392, 200), (1, 8, 8), (129, 1000, 72)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_mma_sync_exact(swz, layout, shape, dtype):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-4, hi=4, seed=M + K)
    C = swz.gemm_mma_sync(A.cuda(), B.cuda(), layout, "serpentine", 2)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("layout", ["naive", "swizzle128", "padded"])
def test_mma_sync_1024(swz, layout):
    A, B = si.gemm_inputs(1024, 1024, 512, "fp16", "uniform", seed=0)
    C = swz.gemm_mma_sync(A.cuda(), B.cuda(), layout, "panel", 4)
    mx, rel = errors(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())
    assert mx <= MAX_ABS and rel <= REL_FRO


def test_mma_sync_4096_sampled(swz):
    A, B = si.gemm_inputs(4096, 4096, 4096, "fp16", "uniform", seed=1)
    C = swz.gemm_mma_sync(A.cuda(), B.cuda(), "swizzle128", "panel", 8)
    ii, jj = si.sample_indices(4096, 4096, 128, 128, 1, seed=2)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    mx, rel = errors(got, ref.gemm_entries_f64(A, B, ii, jj))
    assert mx <= MAX_ABS and rel <= REL_FRO


def test_mma_sync_bad_layouts(swz):
    A = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.float16, device="cuda")
    for lay in [(4, 1, 1, 0), (8, 3, 1, 0), (8, 1, 16, 0), (8, 1, 1, 4), (8, 1, 1, 72)]:
        with pytest.raises(swz.SwzError) as e:
            swz.gemm_mma_sync(A, B, lay)
        assert e.value.code == swz.SWZ_EINVAL
