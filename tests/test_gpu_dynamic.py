"""Dynamic tile scheduler (opts.dynamic): tiles claimed through an atomic
counter instead of work_idx striding.

* Results: exact on small-integer inputs for every tile shape and dtype, and
  bit-identical to the static schedule on real inputs (a tile's K loop does
  not depend on which program runs it).
* Schedule (per-tile trace): every CTA tile is computed exactly once; the
  first wave is the static one (program c takes work index c); each
  program's later work indices increase (they come from one counter) and
  both CTAs of a pair record the same cluster tile and iteration.
* The counter is cleared per launch: back-to-back launches on one workspace
  stay correct.  Misuse is rejected on the host.  A withheld load still ends
  in SWZ_ETIMEOUT with the ring's waits bounded.
"""
import pytest
import torch

import synth_inputs as si
from gpu_util import require_gpu
from oracle import ref
from oracle import tile_order as to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _ws(n=256):
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


CFGS = [dict(tile_n=128), dict(tile_n=256), dict(cta_pair=True)]


@pytest.mark.parametrize("shape", [(768, 640, 576), (300, 392, 200), (1, 8, 8),
                                   (1100, 1304, 136)])
@pytest.mark.parametrize("cfg", CFGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("programs", [0, 4, 6])
def test_exact_integer(swz, shape, cfg, dtype, programs):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-4, hi=4, seed=M + programs)
    ws = _ws()
    C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 2, True, num_programs=programs,
                 dynamic=True, workspace=ws, **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("cfg", CFGS)
def test_tf32_exact(swz, cfg):
    M, N, K = 513, 264, 100
    g = torch.Generator().manual_seed(5)
    A = torch.randint(-8, 9, (M, K), generator=g).float()
    B = torch.randint(-8, 9, (K, N), generator=g).float()
    C = swz.gemm(A.cuda(), B.t().contiguous().cuda(), "panel", 4, True, b_transposed=True,
                 dynamic=True, workspace=_ws(), **cfg)
    swz.check_status()
    assert torch.equal(C.cpu().double(), ref.gemm_f64(A, B))


@pytest.mark.parametrize("cfg", CFGS)
def test_bit_identical_to_static(swz, cfg):
    A, B = si.gemm_inputs(2048, 2048, 1024, "bf16", "normal", seed=4)
    Ad, Bd = A.cuda(), B.cuda()
    ws = _ws()
    C0 = swz.gemm(Ad, Bd, "panel", 8, True, **cfg)
    for _ in range(3):  # back-to-back launches reuse the workspace
        C1 = swz.gemm(Ad, Bd, "panel", 8, True, dynamic=True, workspace=ws, **cfg)
        swz.check_status()
        assert torch.equal(C0, C1)


def _check_trace(trace, gm, gn, order, g, programs, cluster_m):
    """gm x gn CTA tiles, clusters of cluster_m CTAs along M."""
    got = trace.view(gm, gn, 2).cpu().tolist()
    cgm = gm // cluster_m
    ids = to.id_table(order, cgm, gn, g)  # work index of each cluster tile
    static = to.persistent_trace(order, gm, gn, g, programs, cluster_m=cluster_m)
    per_prog = {}
    for m in range(gm):
        for n in range(gn):
            prog, it = got[m][n]
            assert 0 <= prog < programs and it >= 0, (m, n, prog, it)
            assert prog % cluster_m == m % cluster_m  # CTA rank = row within the cluster tile
            if it == 0:
                assert static[(m, n)] == (prog, 0)  # the first wave is static
            per_prog.setdefault(prog, {})
            assert it not in per_prog[prog], "one tile per iteration"
            per_prog[prog][it] = ids[m // cluster_m][n]
    for prog, seq in per_prog.items():
        its = sorted(seq)
        assert its == list(range(len(its)))  # iterations 0, 1, 2, ... without gaps
        ws = [seq[i] for i in its]
        assert ws[0] == prog // cluster_m
        assert all(a < b for a, b in zip(ws, ws[1:]))  # claimed from one counter
        assert all(w >= programs // cluster_m for w in ws[1:])
    if cluster_m == 2:  # both CTAs of a cluster run the same sequence
        for prog in range(0, programs, 2):
            assert per_prog.get(prog) == per_prog.get(prog + 1)


@pytest.mark.parametrize("order,g", [(to.ROW, 1), (to.PANEL, 4), (to.SERPENTINE, 2)])
@pytest.mark.parametrize("programs", [7, 3])
def test_single_cta_trace(swz, order, g, programs):
    A, B = si.gemm_inputs(768, 640, 128, "fp16", "uniform", seed=1)
    trace = torch.full((6 * 5 * 2,), -1, dtype=torch.int32, device="cuda")
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, tile_n=128, num_programs=programs,
                 trace=trace, dynamic=True, workspace=_ws())
    swz.check_status()
    _check_trace(trace, 6, 5, order, g, programs, 1)
    assert torch.equal(C, swz.gemm(A.cuda(), B.cuda(), order, g, True, tile_n=128))


@pytest.mark.parametrize("order,g", [(to.PANEL, 2), (to.SERPENTINE, 2)])
@pytest.mark.parametrize("programs", [4, 6])
def test_pair_trace(swz, order, g, programs):
    A, B = si.gemm_inputs(1536, 1280, 192, "bf16", "uniform", seed=2)
    gm, gn = 12, 5  # CTA tiles of 128 x 256
    trace = torch.full((gm * gn * 2,), -1, dtype=torch.int32, device="cuda")
    swz.gemm(A.cuda(), B.cuda(), order, g, True, cta_pair=True, num_programs=programs,
             trace=trace, dynamic=True, workspace=_ws())
    swz.check_status()
    _check_trace(trace, gm, gn, order, g, programs, 2)


def test_errors(swz):
    A = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    C = torch.empty((256, 256), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ws = _ws(512)

    def call(persistent=1, **kw):
        o = swz.make_opts(dynamic=True, **kw)
        return swz.swz_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 256, 256, 64,
                               swz.SWZ_ROW, 1, persistent, o, s)
    assert call(workspace=ws) == swz.SWZ_OK
    assert call(persistent=0, workspace=ws) == swz.SWZ_EINVAL
    assert call() == swz.SWZ_EINVAL                                  # no workspace
    assert call(workspace=ws[:128]) == swz.SWZ_EINVAL                # too small
    assert call(workspace=ws[16:]) == swz.SWZ_EINVAL                 # misaligned
    assert call(workspace=ws, stream_k=True) == swz.SWZ_EINVAL
    assert call(workspace=ws, smem_swizzle=64) == swz.SWZ_EUNSUPPORTED
    assert swz.workspace_size(256, 256, 64, True, stream_k=False, dynamic=True) == 256
    assert swz.workspace_size(256, 256, 64, False, stream_k=False, dynamic=True) == 0
    swz.check_status()


@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(cta_pair=True)])
def test_withheld_load_times_out_cleanly(swz, cfg):
    A, B = si.gemm_inputs(512, 512, 128, "fp16", "uniform", seed=3)
    Ad, Bd = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    assert swz.swz_check_status(s) == swz.SWZ_OK
    swz.gemm(Ad, Bd, "row", 1, True, debug_flags=swz.SWZ_DEBUG_SKIP_FIRST_LOAD, timeout_ms=50,
             dynamic=True, workspace=_ws(), **cfg)
    assert swz.swz_check_status(s) == swz.SWZ_ETIMEOUT
    C = swz.gemm(Ad, Bd, "row", 1, True, dynamic=True, workspace=_ws(), **cfg)
    swz.check_status()
    assert torch.equal(C, swz.gemm(Ad, Bd, "row", 1, True, **cfg))


def test_dynamic_mode_range(swz):
    A, B = si.gemm_inputs(256, 256, 64, "fp16", "uniform", seed=0)
    with pytest.raises(swz.SwzError) as e:
        swz.gemm(A.cuda(), B.cuda(), "row", 1, True, dynamic=2, workspace=_ws())
    assert e.value.code == swz.SWZ_EINVAL
