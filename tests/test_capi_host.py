"""The C-ABI library builds, loads without a GPU, exports every symbol the
header declares, and its host-only paths (status strings, bijectivity check,
launch planning, argument validation) behave as specified (CPU only)."""
import os
import re

import pytest

from conftest import ROOT
from oracle import tile_order as to


@pytest.fixture(scope="module")
def swz():
    from thread_block_smem_gb300 import build
    build.build()
    import thread_block_smem_gb300 as m
    m.lib()
    return m


def _declared_functions():
    with open(os.path.join(ROOT, "include", "swz.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swz_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(swz):
    declared = _declared_functions()
    assert set(declared) == set(swz.EXPORTS)
    for name in declared:
        assert hasattr(swz.lib(), name), name


def test_strerror(swz):
    for code in range(0, -7, -1):
        assert swz.swz_strerror(code)
    assert swz.swz_strerror(12345) == "unknown status"


@pytest.mark.parametrize("order,gm,gn,g", [
    (to.MORTON, 8, 8, 1), (to.XOR, 8, 8, 1), (to.MORTON, 32, 16, 1), (to.XOR, 32, 16, 1),
    (to.MORTON, 16, 32, 1), (to.XOR, 16, 32, 1), (to.MORTON, 48, 80, 1), (to.XOR, 48, 80, 1),
    (to.PANEL, 48, 80, 16), (to.SERPENTINE, 48, 80, 8), (to.SERPENTINE, 3, 5, 2),
    (to.ROW, 7, 9, 1), (to.COL, 7, 9, 1), (to.MORTON, 3, 3, 1), (to.XOR, 2, 4, 1)])
def test_host_bijectivity_matches_oracle(swz, order, gm, gn, g):
    assert swz.swz_is_bijective(order, gm, gn, g) == int(to.is_bijective(order, gm, gn, g))


def test_bijectivity_rejects_bad_args(swz):
    assert swz.swz_is_bijective(9, 4, 4, 1) == swz.SWZ_EINVAL
    assert swz.swz_is_bijective(to.PANEL, 4, 4, 0) == swz.SWZ_EINVAL
    assert swz.swz_is_bijective(to.ROW, 0, 4, 1) == swz.SWZ_EINVAL


def test_plan_without_device(swz):
    # non-persistent plans and persistent plans with an explicit program
    # count need no device
    assert swz.gemm_plan(1024, 1024, 512, tile_n=128) == (8, 8, 8, 8, 64)
    assert swz.gemm_plan(4096, 4096, 4096, tile_n=256) == (32, 16, 32, 16, 512)
    assert swz.gemm_plan(8192, 8192, 8192, cta_pair=True) == (64, 32, 32, 32, 2048)
    assert swz.gemm_plan(6144, 10240, 4096, tile_n=128) == (48, 80, 48, 80, 3840)
    assert swz.gemm_plan(6100, 10200, 4096, tile_n=128) == (48, 80, 48, 80, 3840)
    assert swz.gemm_plan(8192, 8192, 8192, True, cta_pair=True, num_programs=148) == (
        64, 32, 32, 32, 148)
    assert swz.gemm_plan(300, 392, 200, True, tile_n=256, num_programs=1000) == (3, 2, 3, 2, 6)
    rc, _ = swz.swz_gemm_plan(1024, 1024, 512, 0, swz.make_opts(tile_n=192))
    assert rc == swz.SWZ_EUNSUPPORTED
    # CTA pair with 128-wide tiles: cluster tiles 256 x 128, CTA tiles 128 x 128
    assert swz.gemm_plan(6144, 10240, 4096, cta_pair=True, tile_n=128) == (48, 80, 24, 80, 3840)
    assert swz.gemm_plan(1024, 1024, 512, cta_pair=True, tile_n=128) == (8, 8, 4, 8, 64)
    rc, _ = swz.swz_gemm_plan(1024, 1024, 512, 1, swz.make_opts(cta_pair=True, num_programs=7))
    assert rc == swz.SWZ_EINVAL


def test_stream_k_plan_keeps_every_program(swz):
    # Stream-K shares the tail among all programs: with fewer scheduler units
    # than programs every program stays (each unit's K is split), while the
    # other schedules cap the programs at the units.
    for cfg, units in ((dict(cta_pair=True), 1), (dict(tile_n=128), 4)):
        o = swz.make_opts(num_programs=152, **cfg)
        rc, plan = swz.swz_gemm_plan(256, 256, 1 << 20, 1, o)
        assert rc == swz.SWZ_OK and plan[4] == units * (2 if cfg.get("cta_pair") else 1)
        assert swz.swz_gemm_workspace_size(256, 256, 1 << 20, 1, o) == (swz.SWZ_OK, 0)
        o = swz.make_opts(num_programs=152, stream_k=True, **cfg)
        rc, plan = swz.swz_gemm_plan(256, 256, 1 << 20, 1, o)
        assert rc == swz.SWZ_OK and plan[4] == 152
        rc, n = swz.swz_gemm_workspace_size(256, 256, 1 << 20, 1, o)
        # two slots per CTA: flags (4 words each, 256-byte aligned) and one
        # 128 x tile_n FP32 partial each
        tn = 256 if cfg.get("cta_pair") else 128
        assert rc == swz.SWZ_OK and n == 4864 + 2 * 152 * 128 * tn * 4
    # the same through the Python helper
    assert swz.gemm_plan(256, 256, 1 << 20, True, cta_pair=True, num_programs=152) == (
        2, 1, 1, 1, 2)
    assert swz.gemm_plan(256, 256, 1 << 20, True, cta_pair=True, num_programs=152,
                         stream_k=True) == (2, 1, 1, 1, 152)
    # evenly divided units need no Stream-K workspace
    o = swz.make_opts(num_programs=8, stream_k=True, tile_n=128)
    assert swz.swz_gemm_workspace_size(1024, 1024, 512, 1, o) == (swz.SWZ_OK, 0)


def test_validation_before_device(swz):
    # these are rejected before any CUDA call is made
    E = swz.SWZ_EINVAL
    assert swz.swz_gemm(16, 16, 16, 8, 8, 8, 9, 1, 0) == E           # unknown order
    assert swz.swz_gemm(16, 16, 16, 8, 8, 8, to.PANEL, 0, 0) == E     # group < 1
    assert swz.swz_gemm(0, 16, 16, 8, 8, 8, to.ROW, 1, 0) == E        # null A
    assert swz.swz_gemm(16, 16, 16, 8, 8, 12, to.ROW, 1, 0) == E      # K % 8
    assert swz.swz_gemm(16, 16, 16, 8, 12, 8, to.ROW, 1, 0) == E      # N % 8
    assert swz.swz_gemm(8, 16, 16, 8, 8, 8, to.ROW, 1, 0) == E        # misaligned A
    assert swz.swz_gemm(16, 16, 16, -1, 8, 8, to.ROW, 1, 0) == E      # negative M
    assert swz.swz_gemm(16, 16, 0, 0, 8, 8, to.ROW, 1, 0) == swz.SWZ_OK  # M = 0: no-op
    assert swz.swz_tile_map(9, 4, 4, 1, 16, 16) == E
    assert swz.swz_tile_map(to.ROW, 4, 4, 1, 0, 16) == E
    assert swz.swz_tile_map(to.SERPENTINE, 4, 4, 0, 16, 16) == E
    assert swz.swz_transpose(16, 16, 4, 4, 7) == E                    # unknown layout
    assert swz.swz_transpose(16, 4096, -1, 4, 0) == E
    assert swz.swz_transpose(0, 0, 0, 5, 0) == swz.SWZ_OK             # empty: no-op
    assert swz.swz_transpose(16, 32, 4, 4, 0) == E                    # overlapping
    assert swz.swz_transpose(18, 4096, 4, 4, 0) == E                  # misaligned
    # maximum sizes: the transpose grid's y extent holds 65535 row tiles of
    # 32 (M <= 2,097,120); a GEMM whose tile count does not fit int32 is refused
    assert swz.swz_transpose(16, 1 << 40, 65535 * 32 + 1, 4, 0) == E
    for cfg in (dict(), dict(cta_pair=True), dict(tile_n=128)):
        assert swz.swz_gemm_plan(2**31 - 1, 2**31 - 8, 64, 0, swz.make_opts(**cfg))[0] == E
    rc, plan = swz.swz_gemm_plan(2**20, 2**20, 64, 0, swz.make_opts())
    assert rc == swz.SWZ_OK and plan == (8192, 4096, 8192, 4096, 33554432)


def test_product_does_not_import_oracle():
    # the product package and the bench's product path never name the oracle
    pkg = os.path.join(ROOT, "thread_block_smem_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(from|import)\s+oracle", src, re.M), f
                assert "liboracle" not in src, f
