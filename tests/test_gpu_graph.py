"""CUDA-graph capture and replay of the device-buffer entry points.

Each call is made once eagerly (its kernel variant's one-time set-up), then
recorded with stream capture; the graph is replayed with new operands copied
into the captured buffers before each replay, and every replay must equal the
oracle exactly on small-integer inputs (or bit for bit, for the transpose and
the tile map).  The Stream-K and dynamic-scheduler launches clear device state
before they start (piece flags, the claim counter); these tests check that the
clearing is part of the graph, so that one replay cannot see the previous
replay's state."""
import pytest
import torch

import synth_inputs as si
from gpu_util import capture_graph, require_gpu
from oracle import ref
from oracle import tile_order as to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _replays(swz, g, Ad, Bd, C, M, N, K, dtype, seeds):
    for seed in seeds:
        A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-3, hi=3, seed=seed)
        Ad.copy_(A)
        Bd.copy_(B)
        C.fill_(float("nan"))
        g.replay()
        swz.check_status()
        assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B)), seed


# (M, N, K, dtype, cfg): each static schedule's kernel family once
STATIC = [
    (768, 640, 1024, "bf16", dict(cta_pair=True)),
    (1000, 1000, 520, "fp16", dict(tile_n=256)),
    (768, 640, 512, "fp16", dict(tile_n=128, num_programs=7)),
    (1024, 1024, 512, "bf16", dict(cta_pair=True, tile_n=128, num_programs=8)),
]


@pytest.mark.parametrize("M,N,K,dtype,cfg", STATIC)
def test_graph_static_gemm(swz, M, N, K, dtype, cfg):
    dt = si.torch_dtype(dtype)
    Ad = torch.zeros((M, K), dtype=dt, device="cuda")
    Bd = torch.zeros((K, N), dtype=dt, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g = capture_graph(lambda: swz.gemm(Ad, Bd, "serpentine", 4, True, out=C, **cfg))
    _replays(swz, g, Ad, Bd, C, M, N, K, dtype, seeds=(1, 2, 3))


@pytest.mark.parametrize("M,N,K,cfg", [
    (768, 640, 1024, dict(tile_n=128, num_programs=7)),
    (1280, 1024, 576, dict(cta_pair=True, num_programs=6)),
])
def test_graph_stream_k_workspace(swz, M, N, K, cfg):
    # The flag value a launch waits for is fixed when the call is captured;
    # new operands in every replay make stale partial sums visible.
    n = swz.workspace_size(M, N, K, True, **cfg)
    assert n > 0
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    Ad = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g = capture_graph(lambda: swz.gemm(Ad, Bd, "panel", 2, True, out=C, stream_k=True,
                                       workspace=ws, **cfg))
    _replays(swz, g, Ad, Bd, C, M, N, K, "bf16", seeds=(4, 5, 6, 7))
    # an ordinary call after the replays, on the same workspace
    A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=8)
    Ad.copy_(A)
    Bd.copy_(B)
    swz.gemm(Ad, Bd, "panel", 2, True, out=C, stream_k=True, workspace=ws, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


def test_graph_dynamic(swz):
    M, N, K = 1280, 1024, 576
    cfg = dict(cta_pair=True, num_programs=6, dynamic=True)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    Ad = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.float16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g = capture_graph(lambda: swz.gemm(Ad, Bd, "serpentine", 3, True, out=C, workspace=ws,
                                       **cfg))
    _replays(swz, g, Ad, Bd, C, M, N, K, "fp16", seeds=(9, 10, 11))


def test_graph_gemm_then_transpose(swz):
    # two kernels in one graph: C = A B, then C^T through the XOR-swizzled tile
    M, N, K = 768, 640, 256
    Ad = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Bd = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    Ct = torch.empty((N, M), dtype=torch.float32, device="cuda")

    def step():
        swz.gemm(Ad, Bd, "panel", 4, True, out=C, cta_pair=True)
        swz.transpose(C.view(torch.int32), "xor", out=Ct.view(torch.int32))

    g = capture_graph(step)
    for seed in (12, 13):
        A, B = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-3, hi=3, seed=seed)
        Ad.copy_(A)
        Bd.copy_(B)
        Ct.fill_(float("nan"))
        g.replay()
        swz.check_status()
        want = ref.gemm_f64(A, B).float()
        assert torch.equal(Ct.cpu().view(torch.int32),
                           ref.transpose_u32(want.contiguous().view(torch.int32)))


def test_graph_transpose_and_tile_map(swz):
    M, N = 333, 517
    x = torch.zeros((M, N), dtype=torch.int32, device="cuda")
    y = torch.empty((N, M), dtype=torch.int32, device="cuda")
    g = capture_graph(lambda: swz.transpose(x, "xor", out=y))
    for seed in (14, 15):
        h = si.transpose_input(M, N, seed=seed)
        x.copy_(h)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), ref.transpose_u32(h))

    out = {}

    def maps():
        out["mn"] = swz.tile_map(to.SERPENTINE, 48, 80, 8)

    gm = capture_graph(maps)
    m, n = out["mn"]
    m.fill_(-1)
    n.fill_(-1)
    gm.replay()
    torch.cuda.synchronize()
    assert list(zip(m.tolist(), n.tolist())) == to.tile_sequence(to.SERPENTINE, 48, 80, 8)
