"""ctypes front end of the plain-C oracle (gemm_ref.c) -- test infrastructure.

``build()`` compiles gemm_ref.c with gcc (-O2, no fast-math, no FP
contraction, OpenMP) into oracle/_build/liboracle.so.  The functions below take
CPU torch tensors, widen half-precision inputs to float64 with torch's exact
conversion, and call the C routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (idempotent).  Returns the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
        "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_gemm_rows_f64.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64]
        lib.oracle_gemm_entries_f64.argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, vp]
        lib.oracle_transpose_u32.argtypes = [vp, vp, i64, i64]
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _f64(t: torch.Tensor) -> torch.Tensor:
    return t.detach().to("cpu").to(torch.float64).contiguous()


def gemm_f64(A: torch.Tensor, B: torch.Tensor, row_begin: int = 0,
             row_end: int | None = None) -> torch.Tensor:
    """Rows [row_begin, row_end) of A @ B in float64 (A: M x K, B: K x N)."""
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    row_end = M if row_end is None else row_end
    a, b = _f64(A), _f64(B)
    c = torch.empty((row_end - row_begin, N), dtype=torch.float64)
    _load().oracle_gemm_rows_f64(a.data_ptr(), b.data_ptr(), c.data_ptr(),
                                 M, N, K, row_begin, row_end)
    return c


def gemm_f64_widened(a64: torch.Tensor, b64: torch.Tensor, row_begin: int,
                     row_end: int) -> torch.Tensor:
    """Same as ``gemm_f64`` on inputs already widened to float64 (avoids the
    conversion when the same operands are reused)."""
    M, K = a64.shape
    N = b64.shape[1]
    c = torch.empty((row_end - row_begin, N), dtype=torch.float64)
    _load().oracle_gemm_rows_f64(a64.data_ptr(), b64.data_ptr(), c.data_ptr(),
                                 M, N, K, row_begin, row_end)
    return c


def gemm_entries_f64(A: torch.Tensor, B: torch.Tensor, ii, jj) -> np.ndarray:
    """C[ii[s], jj[s]] in float64 for sampled coordinates."""
    M, K = A.shape
    N = B.shape[1]
    a, b = _f64(A), _f64(B)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    if ii.size and (ii.min() < 0 or ii.max() >= M or jj.min() < 0 or jj.max() >= N):
        raise IndexError("sample outside C")
    out = np.empty(ii.size, dtype=np.float64)
    _load().oracle_gemm_entries_f64(a.data_ptr(), b.data_ptr(), M, N, K,
                                    ii.ctypes.data, jj.ctypes.data, ii.size,
                                    out.ctypes.data)
    return out


def transpose_u32(x: torch.Tensor) -> torch.Tensor:
    """N x M transpose of an M x N int32/uint32 tensor (bit copy)."""
    x = x.detach().to("cpu").contiguous()
    if x.element_size() != 4:
        raise ValueError("32-bit words expected")
    M, N = x.shape
    out = torch.empty((N, M), dtype=x.dtype)
    _load().oracle_transpose_u32(x.data_ptr(), out.data_ptr(), M, N)
    return out
