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


def capture_graph(fn):
    """Run fn once eagerly on a side stream (one-time set-up of the kernels it
    launches), then record it into a torch.cuda.CUDAGraph and return that."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g
