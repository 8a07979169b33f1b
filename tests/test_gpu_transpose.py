"""swz_transpose is bit-identical to the oracle for every shared-memory
layout, at the configured sizes and on ragged and degenerate shapes."""
import pytest
import torch

import synth_inputs as si
from gpu_util import require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


@pytest.mark.parametrize("layout", ["naive", "padded", "xor"])
@pytest.mark.parametrize("shape", [(1024, 2048), (96, 160), (33, 70), (1, 1), (31, 1),
                                   (1, 45), (2048, 1024), (100, 4000)])
def test_transpose_bit_exact(swz, layout, shape):
    M, N = shape
    x = si.transpose_input(M, N, seed=M * 7 + N)
    y = swz.transpose(x.cuda(), layout)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), ref.transpose_u32(x))


def test_transpose_empty(swz):
    x = torch.empty((0, 5), dtype=torch.int32, device="cuda")
    assert swz.transpose(x, "xor").shape == (5, 0)


@pytest.fixture(scope="module")
def full_case():
    # 16384 x 32768 words, 2 GiB each way
    x = si.transpose_input(16384, 32768, seed=11)
    return x, ref.transpose_u32(x)


@pytest.mark.parametrize("layout", ["naive", "padded", "xor"])
def test_transpose_full_size(swz, full_case, layout):
    x, want = full_case
    xd = x.cuda()
    y = swz.transpose(xd, layout)
    torch.cuda.synchronize()
    del xd
    assert torch.equal(y.cpu(), want)
