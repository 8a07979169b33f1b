"""Python binding of libswz.so (include/swz.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; PyTorch supplies device
memory and streams.  There is no fallback: if the library is missing or the
device is not sm_103, calls raise.

Two layers:
  * ``swz_*`` -- one-to-one mirrors of the C entry points (raw device
    pointers as ints, stream as an int cudaStream_t).
  * ``tile_map``, ``gemm``, ``transpose``, ``gemm_plan`` -- the same calls on
    torch tensors (pointers and the current stream are taken from them).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libswz.so")

# status codes and enums (include/swz.h)
SWZ_OK, SWZ_EINVAL, SWZ_ENOTBIJECTIVE, SWZ_EARCH, SWZ_ECUDA, SWZ_ETIMEOUT, SWZ_EUNSUPPORTED = (
    0, -1, -2, -3, -4, -5, -6)
SWZ_ESCRATCH = -7
SWZ_NOALLOC_SCRATCH_BYTES = 40 * 1024 * 1024
SWZ_ROW, SWZ_COL, SWZ_PANEL, SWZ_MORTON, SWZ_XOR, SWZ_SERPENTINE = range(6)
SWZ_F16, SWZ_BF16, SWZ_TF32 = 0, 1, 2
SWZ_B_KN, SWZ_B_NK = 0, 1
SWZ_SMEM_NAIVE, SWZ_SMEM_PADDED, SWZ_SMEM_XOR = 0, 1, 2
SWZ_DEBUG_SKIP_FIRST_LOAD = 1
ORDERS = {"row": SWZ_ROW, "col": SWZ_COL, "panel": SWZ_PANEL, "morton": SWZ_MORTON,
          "xor": SWZ_XOR, "serpentine": SWZ_SERPENTINE}
LAYOUTS = {"naive": SWZ_SMEM_NAIVE, "padded": SWZ_SMEM_PADDED, "xor": SWZ_SMEM_XOR}

EXPORTS = ["swz_tile_map", "swz_is_bijective", "swz_gemm", "swz_gemm_ex", "swz_gemm_plan",
           "swz_transpose", "swz_check_status", "swz_strerror", "swz_last_cuda_error",
           "swz_device_info", "swz_l2_model", "swz_gemm_workspace_size",
           "swz_gemm_streamk_noalloc", "swz_gemm_host", "swz_gemm_mma_sync", "swz_tc_rate",
           "swz_tc_rate_ex",
           "swz_l2_model_bytes", "swz_calibrate", "swz_gemm_die_plan"]


class SwzError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (status {code}, "
                         f"cuda error {swz_last_cuda_error()})")


class swz_gemm_opts(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("tile_n", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("num_programs", ctypes.c_int), ("d_trace", ctypes.c_void_p),
                ("debug_flags", ctypes.c_uint32), ("timeout_ms", ctypes.c_uint32),
                ("stream_k", ctypes.c_int), ("d_workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64), ("b_layout", ctypes.c_int),
                ("smem_swizzle", ctypes.c_int), ("dynamic", ctypes.c_int),
                ("die_split", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libswz.so (built by thread_block_smem_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libswz.so not built ({LIB_PATH}); run "
                               "`python -m thread_block_smem_gb300.build` first")
        L = ctypes.CDLL(LIB_PATH)
        i, vp, u32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32
        ip = ctypes.POINTER(ctypes.c_int)
        L.swz_tile_map.argtypes = [i, i, i, i, vp, vp, vp]
        L.swz_is_bijective.argtypes = [i, i, i, i]
        L.swz_gemm.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
        L.swz_gemm_ex.argtypes = [vp, vp, vp, i, i, i, i, i, i, ctypes.POINTER(swz_gemm_opts), vp]
        L.swz_gemm_plan.argtypes = [i, i, i, i, ctypes.POINTER(swz_gemm_opts), ip, ip, ip, ip, ip]
        L.swz_transpose.argtypes = [vp, vp, i, i, i, vp]
        L.swz_check_status.argtypes = [vp]
        L.swz_strerror.argtypes = [i]
        L.swz_strerror.restype = ctypes.c_char_p
        L.swz_last_cuda_error.argtypes = []
        L.swz_device_info.argtypes = [ip, ip, ip, ip]
        i64p = ctypes.POINTER(ctypes.c_int64)
        L.swz_l2_model.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.c_int64, i, i, i64p, i64p]
        L.swz_l2_model_bytes.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.c_int64, i, i, i, i,
                                         i64p, i64p, i64p]
        L.swz_gemm_workspace_size.argtypes = [i, i, i, i, ctypes.POINTER(swz_gemm_opts),
                                              ctypes.POINTER(ctypes.c_uint64)]
        L.swz_gemm_streamk_noalloc.argtypes = [vp, vp, vp, i, i, i, i, i,
                                               ctypes.POINTER(swz_gemm_opts), vp]
        L.swz_gemm_host.argtypes = [vp, vp, vp, i, i, i, i, i, ctypes.POINTER(swz_gemm_opts),
                                    vp, vp, vp, i, vp]
        L.swz_gemm_mma_sync.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, i, i, vp]
        L.swz_tc_rate.argtypes = [i, i, vp, vp, i, i, vp, vp, vp]
        L.swz_tc_rate_ex.argtypes = [i, i, i, i, vp, vp, i, i, vp, vp, vp]
        L.swz_calibrate.argtypes = [ip, i, ip]
        L.swz_gemm_die_plan.argtypes = [i, i, i, ctypes.POINTER(swz_gemm_opts),
                                        ctypes.POINTER(ctypes.c_int32), i, ip, ip, ip]
        for name in EXPORTS:
            if name != "swz_strerror":
                getattr(L, name).restype = ctypes.c_int
        del u32
        _lib = L
    return _lib


# ---- raw mirrors ------------------------------------------------------------
def swz_tile_map(order, grid_m, grid_n, group, d_m, d_n, stream=0):
    return lib().swz_tile_map(order, grid_m, grid_n, group, d_m, d_n, stream)


def swz_is_bijective(order, grid_m, grid_n, group=1):
    return lib().swz_is_bijective(order, grid_m, grid_n, group)


def swz_gemm(A, B, C, M, N, K, order, group, persistent, stream=0):
    return lib().swz_gemm(A, B, C, M, N, K, order, group, persistent, stream)


def swz_gemm_ex(A, B, C, M, N, K, order, group, persistent, opts, stream=0):
    return lib().swz_gemm_ex(A, B, C, M, N, K, order, group, persistent,
                             ctypes.byref(opts) if opts is not None else None, stream)


def swz_gemm_plan(M, N, K, persistent, opts=None):
    out = [ctypes.c_int(0) for _ in range(5)]
    rc = lib().swz_gemm_plan(M, N, K, persistent,
                             ctypes.byref(opts) if opts is not None else None,
                             *[ctypes.byref(o) for o in out])
    return rc, tuple(o.value for o in out)


def swz_gemm_workspace_size(M, N, K, persistent, opts=None):
    b = ctypes.c_uint64(0)
    rc = lib().swz_gemm_workspace_size(M, N, K, persistent,
                                       ctypes.byref(opts) if opts is not None else None,
                                       ctypes.byref(b))
    return rc, b.value


def swz_gemm_streamk_noalloc(A, B, C, M, N, K, order, group, opts=None, stream=0):
    """Stream-K GEMM without a caller workspace (the library's built-in
    scratch area; see include/swz.h for who needs it and its limits)."""
    return lib().swz_gemm_streamk_noalloc(A, B, C, M, N, K, order, group,
                                          ctypes.byref(opts) if opts is not None else None,
                                          stream)


def swz_calibrate(max_sms=1024):
    """(status, [die of SM id s for s < max_sms], SM count) -- see include/swz.h."""
    dies = (ctypes.c_int * max_sms)()
    n = ctypes.c_int(0)
    rc = lib().swz_calibrate(dies, max_sms, ctypes.byref(n))
    return rc, list(dies[: n.value]), n.value


def swz_gemm_die_plan(M, N, K, opts=None, max_clusters=256):
    """(status, [die << 15 | rank per cluster], P0, U0) of a persistent launch."""
    info = (ctypes.c_int32 * max_clusters)()
    nc, p0, u0 = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().swz_gemm_die_plan(M, N, K, ctypes.byref(opts) if opts is not None else None,
                                 info, max_clusters, ctypes.byref(nc), ctypes.byref(p0),
                                 ctypes.byref(u0))
    return rc, list(info[: nc.value]), p0.value, u0.value


def calibrate():
    """Runs swz_calibrate on the current device; the die of every SM id."""
    rc, dies, _ = swz_calibrate()
    _check(rc, "swz_calibrate")
    return dies


def swz_gemm_host(hA, hB, hC, M, N, K, order, group, opts, dA, dB, dC, slabs=0, stream=0):
    return lib().swz_gemm_host(hA, hB, hC, M, N, K, order, group,
                               ctypes.byref(opts) if opts is not None else None,
                               dA, dB, dC, slabs, stream)


def swz_gemm_mma_sync(A, B, C, M, N, K, dtype, vec, per_phase, max_phase, pad, order, group,
                      stream=0):
    return lib().swz_gemm_mma_sync(A, B, C, M, N, K, dtype, vec, per_phase, max_phase, pad,
                                   order, group, stream)


# named operand layouts of swz_gemm_mma_sync: (vec, per_phase, max_phase, pad)
SMEM_LAYOUTS = {"naive": (8, 1, 1, 0), "padded": (8, 1, 1, 8), "swizzle128": (8, 1, 8, 0),
                "swizzle64": (8, 2, 4, 0)}


def gemm_mma_sync(A, B, layout="swizzle128", order="panel", group=8, out=None, stream=None):
    """C = A @ B through swz_gemm_mma_sync with the given operand layout (a
    name of SMEM_LAYOUTS or a (vec, per_phase, max_phase, pad) tuple)."""
    import torch
    if A.dtype != B.dtype or A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("A and B must both be fp16 or both bf16")
    M, K = A.shape
    N = B.shape[1]
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=A.device)
    lay = SMEM_LAYOUTS[layout] if isinstance(layout, str) else tuple(layout)
    _check(swz_gemm_mma_sync(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                             SWZ_BF16 if A.dtype == torch.bfloat16 else SWZ_F16, *lay,
                             _order(order), group, _stream(stream)), "swz_gemm_mma_sync")
    return C


def swz_tc_rate(dtype, n, A, B, n_mma, num_ctas, d_times, d_D=None, stream=0):
    return lib().swz_tc_rate(dtype, n, A, B, n_mma, num_ctas, d_times, d_D, stream)


def swz_tc_rate_ex(dtype, n, cta_pair, mmas_per_stage, A, B, n_mma, num_ctas, d_times,
                   d_D=None, stream=0):
    return lib().swz_tc_rate_ex(dtype, n, cta_pair, mmas_per_stage, A, B, n_mma, num_ctas,
                                d_times, d_D, stream)


def tc_rate(A, B, n_mma, num_ctas=0, read_acc=False, stream=None, cta_pair=False,
            mmas_per_stage=0):
    """Runs swz_tc_rate_ex on CUDA operand tiles A (128 x 64 fp16/bf16 or
    128 x 32 fp32) and B (n x 64 / n x 32, B stored N x K).  Returns the
    records of the issuing CTAs as a CPU int64 tensor of shape (records, 4)
    -- cycles, ns, SM id, status -- the FLOP one SM does per instruction,
    and CTA 0's accumulator (128 x n fp32 CUDA tensor) when ``read_acc``.
    ``cta_pair``: 2-CTA MMAs of 256 x n; ``mmas_per_stage``: 4, 8 or 16 cuts
    the issue loop into stages as the GEMM's is (0: back to back)."""
    import torch
    code = _dtype_code(A.dtype)
    if B.dtype != A.dtype or not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B: same dtype, contiguous")
    k_row = 128 // A.element_size()
    n = B.shape[0]
    if tuple(A.shape) != (128, k_row) or tuple(B.shape) != (n, k_row):
        raise ValueError("A must be 128 x (128 bytes), B n x (128 bytes)")
    cg = 2 if cta_pair else 1
    ctas = num_ctas or swz_device_info()[1][0] // cg * cg
    times = torch.zeros((ctas // cg, 4), dtype=torch.int64, device=A.device)
    D = torch.zeros((128, n), dtype=torch.float32, device=A.device) if read_acc else None
    _check(swz_tc_rate_ex(code, n, int(bool(cta_pair)), mmas_per_stage, A.data_ptr(),
                          B.data_ptr(), n_mma, ctas, times.data_ptr(),
                          D.data_ptr() if D is not None else None, _stream(stream)),
           "swz_tc_rate_ex")
    k = 8 if code == SWZ_TF32 else 16
    return times.cpu(), 2 * 128 * n * k, D


def swz_transpose(src, dst, M, N, layout, stream=0):
    return lib().swz_transpose(src, dst, M, N, layout, stream)


def swz_check_status(stream=0):
    return lib().swz_check_status(stream)


def swz_strerror(code):
    return lib().swz_strerror(code).decode()


def swz_last_cuda_error():
    return lib().swz_last_cuda_error()


def swz_device_info():
    v = [ctypes.c_int(0) for _ in range(4)]
    rc = lib().swz_device_info(*[ctypes.byref(x) for x in v])
    return rc, tuple(x.value for x in v)


def swz_l2_model(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes, l2_bytes,
                 concurrency, cluster_m=1):
    h, m = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib().swz_l2_model(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes,
                            l2_bytes, concurrency, cluster_m, ctypes.byref(h), ctypes.byref(m))
    return rc, h.value, m.value


def swz_l2_model_bytes(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes, l2_bytes,
                       concurrency, cluster_m=1, l2_partitions=1, k_alternate=0):
    h, m, b = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib().swz_l2_model_bytes(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes,
                                  l2_bytes, l2_partitions, int(k_alternate), concurrency,
                                  cluster_m, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b))
    return rc, h.value, m.value, b.value


def l2_model_predict(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes, l2_bytes,
                     concurrency, cluster_m=1, l2_partitions=1, k_alternate=False):
    """(predicted L2 hit rate in percent, predicted operand DRAM bytes);
    ``l2_partitions`` = 2 is the two-die reading (each half of the L2 keeps
    its own copy of the whole trace), 1 the first page's model;
    ``k_alternate`` replays the K order of the persistent GEMM (odd waves
    descending) instead of the page's ascending one."""
    rc, h, m, b = swz_l2_model_bytes(_order(order), group, M, N, K, tile_m, tile_n, tile_k,
                                     elem_bytes, l2_bytes, concurrency, cluster_m,
                                     l2_partitions, k_alternate)
    _check(rc, "swz_l2_model_bytes")
    return (100.0 * h / (h + m) if h + m else 0.0), b


def l2_model_hit_rate(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes, l2_bytes,
                      concurrency, cluster_m=1):
    """Predicted L2 hit rate (percent) of the offline tile-trace model."""
    rc, h, m = swz_l2_model(_order(order), group, M, N, K, tile_m, tile_n, tile_k, elem_bytes,
                            l2_bytes, concurrency, cluster_m)
    _check(rc, "swz_l2_model")
    return 100.0 * h / (h + m) if h + m else 0.0


strerror = swz_strerror


def _check(rc, what):
    if rc != SWZ_OK:
        raise SwzError(rc, what)


# ---- tensor-level calls -----------------------------------------------------
def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _order(order):
    return ORDERS[order] if isinstance(order, str) else int(order)


def tile_map(order, grid_m, grid_n, group=1, device="cuda", stream=None):
    """Device-computed tile map: (m, n) int32 tensors of length grid_m*grid_n."""
    import torch
    m = torch.empty(grid_m * grid_n, dtype=torch.int32, device=device)
    n = torch.empty_like(m)
    _check(swz_tile_map(_order(order), grid_m, grid_n, group, m.data_ptr(), n.data_ptr(),
                        _stream(stream)), "swz_tile_map")
    return m, n


def make_opts(dtype=SWZ_F16, tile_n=0, cta_pair=False, num_programs=0, trace=None,
              debug_flags=0, timeout_ms=0, stream_k=False, workspace=None,
              b_layout=SWZ_B_KN, smem_swizzle=0, dynamic=False, die_split=False):
    o = swz_gemm_opts()
    o.die_split = 1 if die_split else 0
    o.smem_swizzle = smem_swizzle
    o.dynamic = int(dynamic)
    o.b_layout = b_layout
    o.stream_k = 1 if stream_k else 0
    if workspace is not None:
        o.d_workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    o.dtype = dtype
    o.tile_n = tile_n
    o.cta_pair = 1 if cta_pair else 0
    o.num_programs = num_programs
    o.d_trace = trace.data_ptr() if trace is not None else None
    o.debug_flags = debug_flags
    o.timeout_ms = timeout_ms
    return o


def gemm_plan(M, N, K, persistent=False, tile_n=0, cta_pair=False, num_programs=0,
              stream_k=False):
    """(tiles_m, tiles_n, sched_m, sched_n, programs) of a GEMM launch
    (with ``stream_k`` the program count is not capped at the tile count)."""
    rc, v = swz_gemm_plan(M, N, K, int(bool(persistent)),
                          make_opts(tile_n=tile_n, cta_pair=cta_pair, num_programs=num_programs,
                                    stream_k=stream_k))
    _check(rc, "swz_gemm_plan")
    return v


def workspace_size(M, N, K, persistent=True, tile_n=0, cta_pair=False, num_programs=0,
                   stream_k=True, dynamic=False):
    """Bytes of workspace a Stream-K (or, with dynamic=True and
    stream_k=False, a dynamic-scheduler) launch of this shape needs (0 if
    none)."""
    rc, b = swz_gemm_workspace_size(M, N, K, int(bool(persistent)),
                                    make_opts(tile_n=tile_n, cta_pair=cta_pair,
                                              num_programs=num_programs, stream_k=stream_k,
                                              dynamic=dynamic))
    _check(rc, "swz_gemm_workspace_size")
    return b


def _dtype_code(t):
    import torch
    codes = {torch.float16: SWZ_F16, torch.bfloat16: SWZ_BF16, torch.float32: SWZ_TF32}
    if t not in codes:
        raise TypeError("A and B must be fp16, bf16 or fp32 (TF32)")
    return codes[t]


def gemm(A, B, order="panel", group=8, persistent=False, *, out=None, tile_n=0,
         cta_pair=False, num_programs=0, trace=None, debug_flags=0, timeout_ms=0,
         stream_k=False, workspace=None, b_transposed=False, smem_swizzle=0,
         dynamic=False, die_split=False, stream=None):
    """C = A @ B (fp32) through swz_gemm_ex.  A: M x K; B: K x N, or N x K
    when ``b_transposed`` (B stored transposed); both fp16, both bf16, or both
    fp32 (multiplied as TF32); row-major contiguous CUDA tensors.  fp32 inputs
    need B as N x K: a K x N fp32 B is first transposed on the device with
    swz_transpose (one extra pass over B).  With stream_k, `workspace` is a
    zero-initialised CUDA tensor of at least workspace_size(...) bytes.
    ``smem_swizzle``: swizzle span of the operand stages, 128 (0), 64 or 32.
    ``dynamic``: claim tiles at run time through an atomic counter kept in
    ``workspace`` (a CUDA tensor of at least workspace_size(..., dynamic=True)
    bytes); persistent launches only.  ``die_split``: each die's clusters take
    their own share of the tiles (after ``calibrate()`` on the device)."""
    import torch
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    code = _dtype_code(A.dtype)
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("2-D operands expected")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("row-major contiguous operands expected")
    M, K = A.shape
    if code == SWZ_TF32 and not b_transposed:
        B = transpose(B.view(torch.int32), "xor", stream=stream).view(torch.float32)
        b_transposed = True
    N = B.shape[0] if b_transposed else B.shape[1]
    if (B.shape[1] if b_transposed else B.shape[0]) != K:
        raise ValueError("inner dimensions differ")
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=A.device)
    opts = make_opts(code, tile_n, cta_pair, num_programs, trace, debug_flags, timeout_ms,
                     stream_k, workspace, SWZ_B_NK if b_transposed else SWZ_B_KN,
                     smem_swizzle, dynamic, die_split)
    _check(swz_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _order(order),
                       group, int(bool(persistent)), opts, _stream(stream)), "swz_gemm_ex")
    return C


def gemm_host(hA, hB, hC, dA, dB, dC, order="panel", group=8, *, tile_n=0, cta_pair=False,
              num_programs=0, stream_k=False, workspace=None, slabs=0,
              b_transposed=False, stream=None):
    """C = A @ B from host tensors through swz_gemm_host.  hA (M x K), hB
    (K x N, or N x K when ``b_transposed``; always N x K for fp32 / TF32): CPU
    fp16/bf16/fp32 tensors (pinned for overlap); hC: CPU fp32 M x N;
    dA, dB, dC: CUDA tensors of the same shapes used as staging.  Asynchronous
    on `stream`; synchronise before reading hC."""
    import torch
    M, K = hA.shape
    N = hB.shape[0] if (b_transposed or hA.dtype == torch.float32) else hB.shape[1]
    for t, dev in ((hA, False), (hB, False), (hC, False), (dA, True), (dB, True), (dC, True)):
        if t.is_cuda != dev or not t.is_contiguous():
            raise ValueError("host tensors on the CPU, staging tensors on the GPU, contiguous")
    if hA.dtype != hB.dtype:
        raise TypeError("A and B must have the same dtype")
    code = _dtype_code(hA.dtype)
    opts = make_opts(code, tile_n, cta_pair, num_programs, None, 0, 0, stream_k, workspace,
                     SWZ_B_NK if (b_transposed or code == SWZ_TF32) else SWZ_B_KN)
    _check(swz_gemm_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, _order(order),
                         group, opts, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), slabs,
                         _stream(stream)), "swz_gemm_host")
    return hC


def transpose(x, layout="xor", out=None, stream=None):
    """N x M transpose of an M x N 32-bit CUDA tensor through swz_transpose."""
    import torch
    if x.dim() != 2 or x.element_size() != 4 or not x.is_contiguous():
        raise ValueError("contiguous 2-D tensor of 32-bit words expected")
    M, N = x.shape
    y = out if out is not None else torch.empty((N, M), dtype=x.dtype, device=x.device)
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    _check(swz_transpose(x.data_ptr(), y.data_ptr(), M, N, lay, _stream(stream)),
           "swz_transpose")
    return y


def check_status(stream=None):
    """Raises SwzError(SWZ_ETIMEOUT) if a bounded device wait expired."""
    _check(swz_check_status(_stream(stream)), "swz_check_status")
