"""swz_gemm / swz_gemm_ex against the FP64 oracle.

* exact: small-integer inputs make every product and partial sum exact in
  fp32, so the tensor-core result must equal the oracle bit for bit;
* full compare at the 1024 x 1024 x 512 configuration for every order,
  tile shape, launch mode and the CTA pair;
* sampled compare (entries of every output tile, computed one by one by the
  oracle) at 4096^3, 8192^3 (bf16, CTA pair) and 6144 x 10240 x 4096, in the
  launch configurations the bench times;
* the persistent schedule actually run (per-tile trace) against the oracle's;
* edge cases: ragged M/N/K, K = 0, tiny shapes, non-bijective Morton/XOR.
Tolerance: max |C - Cref| <= 1e-2 and relative Frobenius error <= 1e-3.
"""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref
from oracle import tile_order as to

pytestmark = pytest.mark.gpu

ORDERS_ALL = [(to.ROW, 1), (to.COL, 1), (to.PANEL, 4), (to.MORTON, 1), (to.XOR, 1),
              (to.SERPENTINE, 2)]


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


def _assert_close(got, want, what=""):
    mx, rel = errors(got, want)
    assert mx <= MAX_ABS and rel <= REL_FRO, f"{what}: max abs {mx:.3e}, rel fro {rel:.3e}"


# ---------------------------------------------------------------- exact ----
@pytest.mark.parametrize("shape", [(300, 392, 200), (128, 256, 64), (1, 8, 8), (129, 136, 72),
                                   (513, 264, 1000)])
@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(tile_n=256),
                                 dict(tile_n=256, cta_pair=True)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_integer_inputs_exact(swz, shape, cfg, dtype):
    M, N, K = shape
    A, B = si.small_int_gemm_inputs(M, N, K, dtype, lo=-4, hi=4, seed=M + N + K)
    want = ref.gemm_f64(A, B)
    for persistent in (False, True):
        C = swz.gemm(A.cuda(), B.cuda(), "panel", 2, persistent, **cfg)
        swz.check_status()
        assert torch.equal(C.cpu().double(), want), (shape, cfg, persistent)


# ------------------------------------------------ config 1: full compare ---
@pytest.fixture(scope="module")
def cfg1():
    A, B = si.gemm_inputs(1024, 1024, 512, "fp16", "uniform", seed=0)
    return A.cuda(), B.cuda(), ref.gemm_f64(A, B).numpy()


@pytest.mark.parametrize("order,g", ORDERS_ALL + [(to.PANEL, 1), (to.PANEL, 8), (to.SERPENTINE, 8)])
@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(tile_n=256),
                                 dict(tile_n=256, cta_pair=True)])
def test_cfg1_all_orders(swz, cfg1, order, g, persistent, cfg):
    A, B, want = cfg1
    C = swz.gemm(A, B, order, g, persistent, **cfg)
    swz.check_status()
    _assert_close(C.cpu().numpy(), want, f"order {order} g {g} {cfg}")


@pytest.mark.parametrize("seed", [1, 2])
def test_cfg1_bf16_normal(swz, seed):
    A, B = si.gemm_inputs(1024, 1024, 512, "bf16", "normal", seed=seed)
    want = ref.gemm_f64(A, B).numpy()
    C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 4, True, cta_pair=True)
    swz.check_status()
    _assert_close(C.cpu().numpy(), want)


# ----------------------------------------------- sampled, full-size cases ---
def _sampled(swz, A, B, C, tile_m=128, tile_n=128, per_tile=4, seed=0, what=""):
    M, N = C.shape
    ii, jj = si.sample_indices(M, N, tile_m, tile_n, per_tile, seed)
    want = ref.gemm_entries_f64(A, B, ii, jj)
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].cpu().numpy()
    _assert_close(got, want, what)
    assert torch.isfinite(C).all().item()


@pytest.fixture(scope="module")
def cfg2():
    A, B = si.gemm_inputs(4096, 4096, 4096, "fp16", "uniform", seed=0)
    return A, B, A.cuda(), B.cuda()


CFG2_ORDERS = [(to.ROW, 1), (to.COL, 1), (to.PANEL, 2), (to.PANEL, 4), (to.PANEL, 8),
               (to.PANEL, 16), (to.MORTON, 1), (to.XOR, 1), (to.SERPENTINE, 4),
               (to.SERPENTINE, 8), (to.SERPENTINE, 16)]


@pytest.mark.parametrize("order,g", CFG2_ORDERS)
@pytest.mark.parametrize("persistent", [False, True])
def test_cfg2_4096_fp16(swz, cfg2, order, g, persistent):
    A, B, Ad, Bd = cfg2
    C = swz.gemm(Ad, Bd, order, g, persistent, tile_n=256)
    swz.check_status()
    _sampled(swz, A, B, C, 128, 256, 2, seed=order * 31 + g, what=f"{order}/{g}")


@pytest.fixture(scope="module")
def cfg3():
    A, B = si.gemm_inputs(8192, 8192, 8192, "bf16", "normal", seed=0)
    return A, B, A.cuda(), B.cuda()


@pytest.mark.parametrize("order,g", [(to.PANEL, 4), (to.PANEL, 8), (to.PANEL, 16),
                                     (to.SERPENTINE, 4), (to.SERPENTINE, 8),
                                     (to.SERPENTINE, 16), (to.ROW, 1)])
def test_cfg3_8192_bf16_pair(swz, cfg3, order, g):
    A, B, Ad, Bd = cfg3
    C = swz.gemm(Ad, Bd, order, g, True, cta_pair=True)
    swz.check_status()
    _sampled(swz, A, B, C, 128, 256, 1, seed=order * 17 + g, what=f"{order}/{g}")


@pytest.mark.parametrize("shape", [(6144, 10240, 4096), (6100, 10200, 4096)])
@pytest.mark.parametrize("order,g", [(to.ROW, 1), (to.PANEL, 8), (to.SERPENTINE, 8)])
def test_cfg4_non_power_of_two_grid(swz, shape, order, g):
    M, N, K = shape
    A, B = si.gemm_inputs(M, N, K, "fp16", "uniform", seed=4)
    C = swz.gemm(A.cuda(), B.cuda(), order, g, True, tile_n=128)
    swz.check_status()
    _sampled(swz, A, B, C, 128, 128, 1, seed=g, what=f"{shape} {order}/{g}")


def test_morton_xor_refused_on_non_bijective_grid(swz):
    A = torch.zeros((6144, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 10240), dtype=torch.float16, device="cuda")
    for order in (to.MORTON, to.XOR):
        with pytest.raises(swz.SwzError) as e:
            swz.gemm(A, B, order, 1, False, tile_n=128)
        assert e.value.code == swz.SWZ_ENOTBIJECTIVE


# ------------------------------------------------------------ schedule ---
@pytest.mark.parametrize("order,g", [(to.ROW, 1), (to.PANEL, 4), (to.SERPENTINE, 2),
                                     (to.COL, 1)])
@pytest.mark.parametrize("programs", [0, 7])
def test_single_cta_trace(swz, order, g, programs):
    # 768 x 640 with 128 x 128 tiles: a 6 x 5 grid
    A, B = si.gemm_inputs(768, 640, 128, "fp16", "uniform", seed=1)
    trace = torch.full((6 * 5 * 2,), -1, dtype=torch.int32, device="cuda")
    persistent = programs > 0
    C = swz.gemm(A.cuda(), B.cuda(), order, g, persistent, tile_n=128, num_programs=programs,
                 trace=trace)
    swz.check_status()
    want = to.persistent_trace(order, 6, 5, g, programs if persistent else 30)
    got = trace.view(6, 5, 2).cpu().tolist()
    assert {(m, n): tuple(got[m][n]) for m in range(6) for n in range(5)} == want
    _assert_close(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())


@pytest.mark.parametrize("order,g", [(to.PANEL, 2), (to.SERPENTINE, 2), (to.ROW, 1)])
@pytest.mark.parametrize("programs", [0, 8, 4])
def test_pair_trace(swz, order, g, programs):
    # 768 x 640 with 256 x 256 cluster tiles: 3 x 3 cluster grid (ragged N),
    # 6 x 3 CTA tiles of 128 x 256
    A, B = si.gemm_inputs(768, 640, 192, "bf16", "uniform", seed=2)
    trace = torch.full((6 * 3 * 2,), -1, dtype=torch.int32, device="cuda")
    persistent = programs > 0
    C = swz.gemm(A.cuda(), B.cuda(), order, g, persistent, cta_pair=True,
                 num_programs=programs, trace=trace)
    swz.check_status()
    want = to.persistent_trace(order, 6, 3, g, programs if persistent else 18, cluster_m=2)
    got = trace.view(6, 3, 2).cpu().tolist()
    assert {(m, n): tuple(got[m][n]) for m in range(6) for n in range(3)} == want
    _assert_close(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())


# --------------------------------------------------------------- edges ---
def test_k_zero_and_empty(swz):
    A = torch.empty((64, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((0, 32), dtype=torch.float16, device="cuda")
    C = torch.full((64, 32), 7.0, device="cuda")
    swz.gemm(A, B, "row", 1, False, out=C)
    assert torch.count_nonzero(C).item() == 0
    A = torch.empty((0, 16), dtype=torch.float16, device="cuda")
    B = torch.ones((16, 8), dtype=torch.float16, device="cuda")
    assert swz.gemm(A, B, "row", 1, False).shape == (0, 8)


@pytest.mark.parametrize("shape", [(1, 8, 8), (5, 16, 24), (200, 8, 8), (7, 1000, 16),
                                   (1000, 24, 4104)])
def test_ragged_small(swz, shape):
    M, N, K = shape
    A, B = si.gemm_inputs(M, N, K, "fp16", "uniform", seed=M)
    want = ref.gemm_f64(A, B).numpy()
    for cfg in (dict(tile_n=128), dict(tile_n=256, cta_pair=True)):
        C = swz.gemm(A.cuda(), B.cuda(), "serpentine", 3, True, **cfg)
        swz.check_status()
        _assert_close(C.cpu().numpy(), want, f"{shape} {cfg}")
