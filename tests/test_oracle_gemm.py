"""Pins of the C oracle (FP64 GEMM and transpose) against brute force in
Python integers, closed forms and algebraic identities (CPU only)."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from oracle import ref


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 3), (16, 24, 40), (33, 17, 65)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_small_integer_brute_force(shape, dtype):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-7, hi=7, seed=M + N + K)
    a = [[int(v) for v in row] for row in A.to(torch.int64).tolist()]
    b = [[int(v) for v in row] for row in B.to(torch.int64).tolist()]
    want = [[sum(a[i][k] * b[k][j] for k in range(K)) for j in range(N)] for i in range(M)]
    got = ref.gemm_f64(A, B)
    assert got.tolist() == [[float(v) for v in r] for r in want]


def test_closed_forms():
    K = 37
    ones_a = torch.ones((4, K), dtype=torch.float16)
    ones_b = torch.ones((K, 6), dtype=torch.float16)
    assert torch.equal(ref.gemm_f64(ones_a, ones_b), torch.full((4, 6), float(K), dtype=torch.float64))
    A, B = si.gemm_inputs(9, 9, 9, "fp16", "uniform", seed=3)
    eye = torch.eye(9, dtype=torch.float16)
    assert torch.equal(ref.gemm_f64(eye, B), B.double())
    assert torch.equal(ref.gemm_f64(A, eye), A.double())


def test_transpose_identity_bitwise():
    # (A B)^T = B^T A^T with the same k-ordered sums, so equal bit for bit
    A, B = si.gemm_inputs(13, 21, 34, "bf16", "normal", seed=5)
    lhs = ref.gemm_f64(A, B).T
    rhs = ref.gemm_f64(B.T.contiguous(), A.T.contiguous())
    assert torch.equal(lhs, rhs)


def test_row_slices_and_entries_agree():
    A, B = si.gemm_inputs(40, 30, 50, "fp16", "uniform", seed=2)
    full = ref.gemm_f64(A, B)
    assert torch.equal(ref.gemm_f64(A, B, 7, 19), full[7:19])
    ii, jj = si.sample_indices(40, 30, 16, 16, 3, seed=1)
    got = ref.gemm_entries_f64(A, B, ii, jj)
    assert np.array_equal(got, full.numpy()[ii, jj])


def test_against_rational_sum():
    # exact rational sum of the fp16 products, rounded once, vs the oracle:
    # the only rounding in the oracle is the double accumulation.
    from fractions import Fraction
    A, B = si.gemm_inputs(3, 4, 300, "fp16", "uniform", seed=9)
    a, b = A.double().tolist(), B.double().tolist()
    got = ref.gemm_f64(A, B).tolist()
    for i in range(3):
        for j in range(4):
            exact = sum(Fraction(a[i][k]) * Fraction(b[k][j]) for k in range(300))
            assert abs(got[i][j] - float(exact)) <= 300 * 2.0**-52 * max(1.0, abs(float(exact)))


def test_half_widening_known_bits():
    bits16 = torch.tensor([0x3C00, 0xC000, 0x0001, 0x7BFF], dtype=torch.int32).to(torch.int16)
    h = bits16.view(torch.float16).double().tolist()
    assert h == [1.0, -2.0, 2.0**-24, 65504.0]
    bb = torch.tensor([0x3F80, 0xC040], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().tolist()
    assert bb == [1.0, -3.0]


def test_transpose_oracle():
    x = torch.tensor([[1, 2, 3], [4, 5, 6]], dtype=torch.int32)
    assert ref.transpose_u32(x).tolist() == [[1, 4], [2, 5], [3, 6]]
    y = si.transpose_input(64, 96, seed=4)
    t = ref.transpose_u32(y)
    assert t.shape == (96, 64)
    assert torch.equal(ref.transpose_u32(t), y)
    assert np.array_equal(t.numpy(), y.numpy().T)
