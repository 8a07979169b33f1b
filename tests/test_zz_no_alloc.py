"""swz_gemm_streamk_noalloc: the Stream-K GEMM for callers that cannot
allocate device memory (they only hold their inputs and outputs, e.g. plugin
hosts that own every allocation or loops where cudaMalloc's device-wide
synchronisation is not acceptable).  It uses the library's built-in scratch
area instead of a caller workspace, so its output must match the workspace
entry point (swz_gemm_ex with stream_k) on the same inputs -- checked on two
calls in a row, the second after the first has left its contents in the
shared scratch area.  This file is collected last on purpose."""
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
        A, B = A.cuda(), B.cuda()
        want = _with_workspace(swz, A, B, order, group, **cfg)
        got = _noalloc(swz, A, B, order, group, **cfg)
        mx, rel = errors(got.cpu().numpy(), want.cpu().numpy())
        assert mx <= MAX_ABS and rel <= REL_FRO, (call, mx, rel)


def test_noalloc_rejects_launch_beyond_scratch(swz):
    # 4000 programs x 128 x 128 fp32 partials would need ~262 MB of scratch
    A = torch.zeros((8192, 128), dtype=torch.float16, device="cuda")
    B = torch.zeros((128, 8192), dtype=torch.float16, device="cuda")
    C = torch.empty((8192, 8192), dtype=torch.float32, device="cuda")
    opts = swz.make_opts(tile_n=128, num_programs=4000)
    rc = swz.swz_gemm_streamk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), 8192, 8192, 128,
                                      swz.SWZ_ROW, 1, opts, _stream())
    assert rc == swz.SWZ_ESCRATCH
    assert "scratch" in swz.swz_strerror(rc)


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
