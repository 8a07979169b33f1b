"""Bounded waits: with the first operand load withheld, the consumer's wait
expires after its bound, the kernel records SWZ_ETIMEOUT, releases TMEM and
returns; the host reads the status once and the context stays usable.  No
fault, trap or unbounded wait is involved."""
import pytest
import torch

import synth_inputs as si
from gpu_util import MAX_ABS, REL_FRO, errors, require_gpu
from oracle import ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    return require_gpu()


@pytest.mark.parametrize("cfg", [dict(tile_n=128), dict(tile_n=256),
                                 dict(tile_n=256, cta_pair=True)])
def test_withheld_load_times_out_cleanly(swz, cfg):
    A, B = si.gemm_inputs(256, 512, 128, "fp16", "uniform", seed=3)
    Ad, Bd = A.cuda(), B.cuda()
    assert swz.swz_check_status(torch.cuda.current_stream().cuda_stream) == swz.SWZ_OK
    swz.gemm(Ad, Bd, "row", 1, False, debug_flags=swz.SWZ_DEBUG_SKIP_FIRST_LOAD,
             timeout_ms=50, **cfg)
    s = torch.cuda.current_stream().cuda_stream
    assert swz.swz_check_status(s) == swz.SWZ_ETIMEOUT
    assert swz.swz_check_status(s) == swz.SWZ_OK  # read once, then cleared
    # the context is intact: a normal launch right after is correct
    C = swz.gemm(Ad, Bd, "row", 1, True, **cfg)
    swz.check_status()
    mx, rel = errors(C.cpu().numpy(), ref.gemm_f64(A, B).numpy())
    assert mx <= MAX_ABS and rel <= REL_FRO
