"""Helpers shared by the GPU tests (no arithmetic of the method here)."""
import numpy as np
import torch


def require_gpu():
    import thread_block_smem_gb300 as swz
    from thread_block_smem_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    rc, (sms, l2, major, minor) = swz.swz_device_info()
    assert rc == 0 and (major, minor) == (10, 3), (rc, major, minor)
    return swz


def errors(got, want):
    """(max abs error, relative Frobenius error) of float arrays."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    d = got - want
    denom = np.linalg.norm(want)
    return float(np.abs(d).max()) if d.size else 0.0, float(np.linalg.norm(d) / denom) if denom else float(np.linalg.norm(d))


# GEMM tolerance of the specification: max |C - Cref| <= 1e-2 and
# ||C - Cref||_F / ||Cref||_F <= 1e-3.
MAX_ABS = 1e-2
REL_FRO = 1e-3
