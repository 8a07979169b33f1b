"""GEMMs back to back in one stream.  Every GEMM launch allows programmatic
dependent launch: a GEMM may start its prologue while the previous kernel of
the stream finishes, and touches global memory only after that kernel has
completed.  So:

* read after write: a GEMM that reads the previous GEMM's output sees all of
  it (the output is filled with NaN before every round);
* write after read: a GEMM that overwrites the previous GEMM's input does so
  only after that GEMM has read it;

eagerly and replayed from a CUDA graph.  The first GEMM of each pair covers a
few tiles, so the second one's CTAs find free SMs at once.  Inputs are small
integers: the first products stay below 2^11, exact in TF32 when the second
GEMM reads them as fp32 operands, and every sum stays below 2^24."""
import pytest
import torch

import synth_inputs as si
from gpu_util import capture_graph, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu

CFGS = [dict(tile_n=128), dict(cta_pair=True)]


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _ints(shape, lo, hi, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


@pytest.mark.parametrize("cfg", CFGS)
def test_read_after_write(swz, cfg):
    # C1 = A B over a long K on 8 or fewer tiles, then C2 = C1 B2 (TF32)
    M, K, N, N2 = 256, 1024, 384, 256
    A = _ints((M, K), -1, 1, 1, torch.float16)
    B = _ints((K, N), -1, 1, 2, torch.float16)
    B2t = _ints((N2, N), -2, 2, 3, torch.float32)  # B2 stored N2 x N (K-major)
    want1 = ref.gemm_f64(A, B)
    assert want1.abs().max().item() < 2 ** 11
    want2 = want1 @ B2t.double().t()
    Ad, Bd, B2d = A.cuda(), B.cuda(), B2t.cuda()
    C1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C2 = torch.empty((M, N2), dtype=torch.float32, device="cuda")

    def pair():
        C1.fill_(float("nan"))
        swz.gemm(Ad, Bd, "row", 1, True, out=C1, **cfg)
        swz.gemm(C1, B2d, "row", 1, True, out=C2, b_transposed=True, **cfg)

    for _ in range(3):
        C2.fill_(float("nan"))
        pair()
        swz.check_status()
        assert torch.equal(C1.cpu().double(), want1)
        assert torch.equal(C2.cpu().double(), want2)
    g = capture_graph(pair)
    for _ in range(3):
        C2.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        swz.check_status()
        assert torch.equal(C2.cpu().double(), want2)


@pytest.mark.parametrize("cfg", CFGS)
def test_write_after_read(swz, cfg):
    # C1 = X B (TF32, 4 tiles, K = 4096), then X = Y Z overwrites X
    M, K, N = 256, 4096, 256
    X0 = _ints((M, K), -1, 1, 4, torch.float32)
    Bt = _ints((N, K), -1, 1, 5, torch.float32)  # B stored N x K
    Y, Z = si.small_int_gemm_inputs(M, K, 64, "fp16", lo=-2, hi=2, seed=6)
    want1 = X0.double() @ Bt.double().t()
    wantx = ref.gemm_f64(Y, Z)
    Bd, Yd, Zd = Bt.cuda(), Y.cuda(), Z.cuda()
    X = torch.empty((M, K), dtype=torch.float32, device="cuda")
    X0d = X0.cuda()
    C1 = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def pair():
        X.copy_(X0d)
        swz.gemm(X, Bd, "row", 1, True, out=C1, b_transposed=True, **cfg)
        swz.gemm(Yd, Zd, "row", 1, True, out=X, **cfg)

    for _ in range(3):
        C1.fill_(float("nan"))
        pair()
        swz.check_status()
        assert torch.equal(C1.cpu().double(), want1)
        assert torch.equal(X.cpu().double(), wantx)
    g = capture_graph(pair)
    for _ in range(3):
        C1.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        swz.check_status()
        assert torch.equal(C1.cpu().double(), want1)
        assert torch.equal(X.cpu().double(), wantx)


@pytest.mark.parametrize("cfg,programs", [(dict(tile_n=128), 7), (dict(cta_pair=True), 6)])
def test_schedulers_with_state_back_to_back(swz, cfg, programs):
    # Stream-K launches sharing one workspace and dynamic-scheduler launches
    # sharing one counter, enqueued back to back with no synchronisation,
    # then a TF32 Stream-K GEMM reading the first result: every result exact
    M, N, K = 768, 640, 1024
    A1, B1 = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=21)
    A2, B2 = si.small_int_gemm_inputs(M, N, K, "bf16", lo=-1, hi=1, seed=22)
    B3t = _ints((256, N), -2, 2, 23, torch.float32)
    w1, w2 = ref.gemm_f64(A1, B1), ref.gemm_f64(A2, B2)
    w3 = w1 @ B3t.double().t()
    d = [X.cuda() for X in (A1, B1, A2, B2)]
    n = swz.workspace_size(M, N, K, True, num_programs=programs, **cfg)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    n3 = swz.workspace_size(M, 256, N, True, num_programs=programs, **cfg)
    ws3 = torch.zeros(max(n3, 256), dtype=torch.uint8, device="cuda")
    wd = torch.zeros(256, dtype=torch.uint8, device="cuda")
    sk = dict(persistent=True, num_programs=programs, stream_k=True, **cfg)
    dyn = dict(persistent=True, num_programs=programs, dynamic=True, workspace=wd, **cfg)
    for _ in range(2):
        C1 = swz.gemm(d[0], d[1], "panel", 2, workspace=ws, **sk)
        C2 = swz.gemm(d[2], d[3], "panel", 2, workspace=ws, **sk)
        C3 = swz.gemm(d[0], d[1], "serpentine", 2, **dyn)
        C4 = swz.gemm(d[2], d[3], "serpentine", 2, **dyn)
        C5 = swz.gemm(C1, B3t.cuda(), "row", 1, b_transposed=True, workspace=ws3, **sk)
        swz.check_status()
        for C, want in ((C1, w1), (C2, w2), (C3, w1), (C4, w2), (C5, w3)):
            assert torch.equal(C.cpu().double(), want)
