"""swz_gemm_streamk_noalloc: the Stream-K GEMM for callers that cannot
allocate device memory (they only hold their inputs and outputs, e.g. plugin
hosts that own every allocation or loops where cudaMalloc's device-wide
synchronisation is not acceptable).  It uses the library's built-in scratch
area instead of a caller workspace.  Both entry points run the same
deterministic kernel, so its output must equal the workspace entry point's
(swz_gemm_ex with stream_k) bit for bit -- checked on two calls in a row, the
second after the first has left its contents in the shared scratch area --
and the oracle's, exactly on integer inputs and within the GEMM tolerance on
sampled entries at 8192^3.  This file is collected last on purpose."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, capture_graph, errors, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc(swz, A, B, order, group, **cfg):
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    opts = swz.make_opts(swz.SWZ_BF16 if A.dtype == torch.bfloat16 else swz.SWZ_F16, **cfg)
    rc = swz.swz_gemm_streamk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                      swz.ORDERS[order], group, opts, _stream())
    assert rc == swz.SWZ_OK, swz.swz_strerror(rc)
    assert swz.swz_check_status(_stream()) == swz.SWZ_OK
    return C


def _with_workspace(swz, A, B, order, group, **cfg):
    M, K = A.shape
    N = B.shape[1]
    n = swz.workspace_size(M, N, K, True, **cfg)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    C = swz.gemm(A, B, order, group, True, stream_k=True, workspace=ws, **cfg)
    swz.check_status()
    return C


@pytest.mark.parametrize("M,N,K,dtype,order,group,cfg", [
    (768, 640, 1024, "fp16", "panel", 2, dict(tile_n=128, num_programs=7)),
    (1280, 1024, 576, "bf16", "serpentine", 3, dict(cta_pair=True, num_programs=6)),
    (8192, 8192, 8192, "bf16", "panel", 8, dict(cta_pair=True)),
])
def test_noalloc_matches_workspace_entry_point_twice(swz, M, N, K, dtype, order, group, cfg):
    for call, seed in enumerate((11, 12)):
        A, B = si.gemm_inputs(M, N, K, dtype, "normal" if dtype == "bf16" else "uniform",
                              seed=seed)
        Ad, Bd = A.cuda(), B.cuda()
        want = _with_workspace(swz, Ad, Bd, order, group, **cfg)
        got = _noalloc(swz, Ad, Bd, order, group, **cfg)
        assert torch.equal(got, want), call
        # and against the oracle: every entry on the small shapes, sampled
        # rows and columns of every tile row at 8192^3
        if M * N <= 1 << 20:
            wantf = ref.gemm_f64(A, B).numpy()
            mx, rel = errors(got.cpu().numpy(), wantf)
        else:
            ii, jj = si.sample_indices(M, N, 128, 256, 1, seed=seed)
            wantf = ref.gemm_entries_f64(A, B, ii, jj)
            gotf = got[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
            mx, rel = errors(gotf, wantf)
        assert mx <= MAX_ABS and rel <= REL_FRO, (call, mx, rel)


def test_noalloc_exact_on_integer_inputs(swz):
    # small-integer operands: every partial sum is an integer below 2^24, so
    # FP32 accumulation in any order gives the FP64 result exactly
    M, N, K = 1280, 1024, 576
    for seed in (31, 32):
        A, B = si.small_int_gemm_inputs(M, N, K, "fp16", lo=-4, hi=4, seed=seed)
        got = _noalloc(swz, A.cuda(), B.cuda(), "serpentine", 2, tile_n=256, num_programs=12)
        assert torch.equal(got.cpu().double(), ref.gemm_f64(A, B)), seed


def test_noalloc_scratch_holds_the_largest_default_launch(swz):
    # the default program count (the resident capacity) with the widest
    # tiles: two workspace slots per program of 128 x 256 FP32 partials
    rc, (sms, _, _, _) = swz.swz_device_info()
    assert rc == swz.SWZ_OK
    for cfg in (dict(tile_n=256), dict(cta_pair=True)):
        _, (_, _, _, _, P) = swz.swz_gemm_plan(4096, 4096, 4096, 1,
                                               swz.make_opts(stream_k=True, **cfg))
        n = swz.workspace_size(4096, 4096, 4096, True, **cfg)
        flags = (2 * P * 16 + 255) // 256 * 256
        assert n == flags + 2 * P * 128 * 256 * 4, (cfg, P, n)
        assert n <= swz.SWZ_NOALLOC_SCRATCH_BYTES, (cfg, P, n)


def test_noalloc_scratch_boundary(swz):
    # 128-wide tiles: each program needs 2 x 64 KB of partial sums and 32
    # bytes of flags.  319 programs fit in the scratch area (the launch is
    # then refused only because 319 programs cannot all be resident); 320 do
    # not, and are refused for the scratch area before anything else.
    M = N = 8192
    K = 128
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    limit = swz.SWZ_NOALLOC_SCRATCH_BYTES
    sizes = {P: swz.workspace_size(M, N, K, True, tile_n=128, num_programs=P) for P in (319, 320)}
    assert sizes[319] <= limit < sizes[320]
    for P, want in ((319, swz.SWZ_EUNSUPPORTED), (320, swz.SWZ_ESCRATCH)):
        opts = swz.make_opts(tile_n=128, num_programs=P)
        rc = swz.swz_gemm_streamk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                          swz.SWZ_ROW, 1, opts, _stream())
        assert rc == want, (P, swz.swz_strerror(rc))
    assert "scratch" in swz.swz_strerror(swz.SWZ_ESCRATCH)


def test_noalloc_graph_replay(swz):
    # the flag clearing is recorded with the launch, so every replay of the
    # captured call starts from clear flags; new operands in every replay
    M, N, K = 1280, 1024, 576
    Ad = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    opts = swz.make_opts(swz.SWZ_BF16, cta_pair=True, num_programs=6)

    def call():
        rc = swz.swz_gemm_streamk_noalloc(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), M, N, K,
                                          swz.SWZ_PANEL, 2, opts, _stream())
        assert rc == swz.SWZ_OK, swz.swz_strerror(rc)

    g = capture_graph(call)
    for seed in (21, 22, 23):
        A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=seed)
        Ad.copy_(A)
        Bd.copy_(B)
        C.fill_(float("nan"))
        g.replay()
        assert swz.swz_check_status(_stream()) == swz.SWZ_OK
        assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B)), seed
