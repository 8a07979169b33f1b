"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
arithmetic of the GEMM, the tile orders or the transpose.  Both the CUDA path
and the CPU oracle receive exactly the tensors returned here (the half-precision
values are rounded once, here, and both sides read those same bits).

Recipes (workload shapes come from the benchmark in Lei Mao, "CUDA Thread Block
Swizzle", section "CUDA Thread Block Swizzle Benchmark", and the transpose case
study in "CUDA Swizzle & bank conflict", section "Matrix Transpose"):

* ``gemm_inputs``: one CPU ``torch.Generator`` seeded with ``seed``; A (M x K)
  is drawn first, then B (K x N) from the same stream.  ``dist="uniform"``
  draws U[-1, 1) as ``2*rand-1``; ``dist="normal"`` draws N(0, 1).  The fp32
  draw is then rounded to fp16 or bf16 (round to nearest even).
* ``small_int_gemm_inputs``: integers drawn uniformly from [lo, hi]; exactly
  representable in fp16/bf16 for |v| <= 256.
* ``transpose_input``: uniform 32-bit words from numpy's PCG64 seeded with
  ``seed``, returned as an int32 tensor holding the raw bits.
"""
from __future__ import annotations

import numpy as np
import torch

_DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def gemm_inputs(M: int, N: int, K: int, dtype: str = "fp16",
                dist: str = "uniform", seed: int = 0):
    """Return CPU tensors (A[M,K], B[K,N]) in ``dtype``, row-major, contiguous."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if dist == "uniform":
        a = torch.rand((M, K), generator=g, dtype=torch.float32) * 2.0 - 1.0
        b = torch.rand((K, N), generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        a = torch.randn((M, K), generator=g, dtype=torch.float32)
        b = torch.randn((K, N), generator=g, dtype=torch.float32)
    else:
        raise ValueError(f"unknown dist {dist!r}")
    return a.to(_DT[dtype]).contiguous(), b.to(_DT[dtype]).contiguous()


def small_int_gemm_inputs(M: int, N: int, K: int, dtype: str = "fp16",
                          lo: int = -4, hi: int = 4, seed: int = 0):
    """Integer-valued A, B (exact in half precision) for exact-sum checks."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    a = torch.randint(lo, hi + 1, (M, K), generator=g, dtype=torch.int64)
    b = torch.randint(lo, hi + 1, (K, N), generator=g, dtype=torch.int64)
    return a.to(_DT[dtype]).contiguous(), b.to(_DT[dtype]).contiguous()


def transpose_input(M: int, N: int, seed: int = 0) -> torch.Tensor:
    """M x N matrix of uniform random 32-bit words (int32 tensor of raw bits)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    words = rng.integers(0, 2**32, size=(M, N), dtype=np.uint32)
    return torch.from_numpy(words.view(np.int32))


def sample_indices(M: int, N: int, per_tile_m: int, per_tile_n: int,
                   samples_per_tile: int, seed: int = 0):
    """Random (i, j) output coordinates: ``samples_per_tile`` in every
    per_tile_m x per_tile_n block of an M x N output (ragged edge blocks
    included), plus the four corners.  Returns two int64 numpy arrays."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    ii, jj = [], []
    for m0 in range(0, M, per_tile_m):
        hm = min(per_tile_m, M - m0)
        for n0 in range(0, N, per_tile_n):
            hn = min(per_tile_n, N - n0)
            ii.append(m0 + rng.integers(0, hm, size=samples_per_tile))
            jj.append(n0 + rng.integers(0, hn, size=samples_per_tile))
    ii.append(np.array([0, 0, M - 1, M - 1]))
    jj.append(np.array([0, N - 1, 0, N - 1]))
    return (np.concatenate(ii).astype(np.int64),
            np.concatenate(jj).astype(np.int64))


def device_words(M: int, N: int, seed: int = 0, device: str = "cuda") -> torch.Tensor:
    """M x N int32 tensor of random words in [0, 2^31) drawn on `device` by
    torch's generator for that device (for sizes too large to draw on the
    host); reproducible for a given seed on one kind of device."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.empty((M, N), dtype=torch.int32, device=device).random_(generator=g)
