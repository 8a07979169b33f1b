"""swz_tc_rate: the tensor-core rate measurement does the MMA work it counts.

* The accumulator CTA 0 reads back equals (n_mma / 4) * A * B^T exactly on
  small-integer operands (exact in fp16, bf16 and TF32; every partial sum is
  an integer far below 2^24), for every dtype and MMA width.
* A rate run on every SM completes, lands one CTA per SM, and yields a
  FLOP-per-clock figure and an SM clock in plausible ranges; TF32 retires
  fewer FLOP per clock than fp16.
"""
import pytest
import torch

from gpu_util import require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


TORCH_DT = {"fp16": torch.float16, "bf16": torch.bfloat16, "tf32": torch.float32}


def _operands(dtype, n, seed):
    g = torch.Generator().manual_seed(seed)
    k_row = 32 if dtype == "tf32" else 64  # 128-byte rows
    A = torch.randint(-4, 5, (128, k_row), generator=g).to(TORCH_DT[dtype])
    B = torch.randint(-4, 5, (n, k_row), generator=g).to(TORCH_DT[dtype])
    return A, B


@pytest.mark.parametrize("n", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16", "tf32"])
@pytest.mark.parametrize("n_mma", [4, 12])
def test_accumulator_exact(swz, dtype, n, n_mma):
    A, B = _operands(dtype, n, seed=n + n_mma)
    times, flop, D = swz.tc_rate(A.cuda(), B.cuda(), n_mma, num_ctas=2, read_acc=True)
    assert (times[:, 3] == 0).all()
    want = ref.gemm_f64(A, B.t().contiguous()) * (n_mma // 4)
    assert torch.equal(D.cpu().double(), want)
    assert flop == 2 * 128 * n * (8 if dtype == "tf32" else 16)


def test_rate_all_sms(swz):
    sms = swz.swz_device_info()[1][0]
    rates = {}
    for dtype in ("bf16", "fp16", "tf32"):
        A, B = _operands(dtype, 256, seed=1)
        swz.tc_rate(A.cuda(), B.cuda(), 256)  # warm-up
        times, flop, _ = swz.tc_rate(A.cuda(), B.cuda(), 8192)
        assert times.shape == (sms, 4)
        assert (times[:, 3] == 0).all()
        assert len(set(times[:, 2].tolist())) == sms  # one CTA per SM
        cyc, ns = times[:, 0].double(), times[:, 1].double()
        fpc = (8192 * flop / cyc).median().item()
        mhz = (cyc / ns * 1e3).median().item()
        assert 300.0 < mhz < 2600.0, mhz
        rates[dtype] = fpc
    assert 1024 <= rates["bf16"] <= 32768, rates
    assert abs(rates["bf16"] / rates["fp16"] - 1.0) < 0.05, rates
    assert rates["tf32"] < rates["fp16"], rates


def test_tc_rate_errors(swz):
    A, B = _operands("bf16", 256, seed=2)
    Ad, Bd = A.cuda(), B.cuda()
    t = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    sms = swz.swz_device_info()[1][0]
    args = dict(A=Ad.data_ptr(), B=Bd.data_ptr(), d_times=t.data_ptr(), stream=s)
    assert swz.swz_tc_rate(swz.SWZ_BF16, 96, n_mma=4, num_ctas=1, **args) == swz.SWZ_EINVAL
    assert swz.swz_tc_rate(swz.SWZ_BF16, 256, n_mma=0, num_ctas=1, **args) == swz.SWZ_EINVAL
    assert swz.swz_tc_rate(swz.SWZ_BF16, 256, n_mma=(1 << 24) + 1, num_ctas=1,
                           **args) == swz.SWZ_EINVAL
    assert swz.swz_tc_rate(swz.SWZ_BF16, 256, n_mma=4, num_ctas=sms + 1,
                           **args) == swz.SWZ_EINVAL
    assert swz.swz_tc_rate(7, 256, n_mma=4, num_ctas=1, **args) == swz.SWZ_EINVAL
    assert swz.swz_tc_rate(swz.SWZ_BF16, 256, Ad.data_ptr() + 8, Bd.data_ptr(), 4, 1,
                           t.data_ptr(), None, s) == swz.SWZ_EINVAL


@pytest.mark.parametrize("n", [128, 256])
@pytest.mark.parametrize("stage", [0, 4, 8, 16])
@pytest.mark.parametrize("pair", [False, True])
def test_pair_and_stage_modes_exact(swz, n, stage, pair):
    # a pair's MMA is 256 x n: CTA 0 holds rows 0..127 of the accumulator and
    # B's columns come half from each CTA; stages change only the issue loop
    A, B = _operands("bf16", n, seed=n + stage)
    n_mma = 32
    times, flop, D = swz.tc_rate(A.cuda(), B.cuda(), n_mma, num_ctas=4, read_acc=True,
                                 cta_pair=pair, mmas_per_stage=stage)
    assert times.shape == ((2 if pair else 4), 4)
    assert (times[:, 3] == 0).all()
    assert torch.equal(D.cpu().double(), ref.gemm_f64(A, B.t().contiguous()) * (n_mma // 4))


def test_stage_loop_rates(swz):
    # back to back, a pair's MMAs run at the one-CTA rate per SM; cutting the
    # loop into stages never makes it faster than that, and stages of 16
    # 128-wide MMAs keep at least 90 % of it
    A, B = _operands("bf16", 256, seed=5)
    Ad, Bd = A.cuda(), B.cuda()
    swz.tc_rate(Ad, Bd, 1024)  # warm-up

    def fpc(n, pair, stage):
        t, flop, _ = swz.tc_rate(Ad, Bd[:n].contiguous(), 16384, cta_pair=pair,
                                 mmas_per_stage=stage)
        assert (t[:, 3] == 0).all()
        return (16384 * flop / t[:, 0].double()).median().item()

    base = fpc(256, False, 0)
    assert abs(fpc(256, True, 0) / base - 1.0) < 0.03
    for stage in (4, 8, 16):
        assert fpc(128, True, stage) <= base * 1.03
    assert fpc(128, True, 16) >= 0.9 * base


def test_tc_rate_ex_errors(swz):
    A, B = _operands("bf16", 256, seed=2)
    Ad, Bd = A.cuda(), B.cuda()
    t = torch.zeros(4 * 4, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    E, U = swz.SWZ_EINVAL, swz.SWZ_EUNSUPPORTED

    def call(dtype=swz.SWZ_BF16, n=256, pair=0, stage=0, n_mma=16, ctas=2):
        return swz.swz_tc_rate_ex(dtype, n, pair, stage, Ad.data_ptr(), Bd.data_ptr(), n_mma,
                                  ctas, t.data_ptr(), None, s)

    assert call(stage=5) == E
    assert call(stage=8, n_mma=12) == E        # not a whole number of stages
    assert call(pair=2) == E
    assert call(pair=1, n=64) == E             # a pair's MMA is 128 or 256 wide
    assert call(pair=1, ctas=3) == E           # whole pairs only
    assert call(dtype=swz.SWZ_TF32, pair=1) == U
    assert call(dtype=swz.SWZ_TF32, stage=4) == U
    assert call() == swz.SWZ_OK
    swz.check_status()
