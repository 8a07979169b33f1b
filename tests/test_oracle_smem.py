"""Pins of the shared-memory oracle: the second page's Triton tables and
transpose conflict arithmetic, swizzle invariants and closed forms (CPU)."""
import pytest

from conftest import read_lines
from oracle import smem_bank as sb


def _triton_tables():
    out, cur = [], None
    for ln in read_lines("sbc_triton_tables.txt"):
        if ln[0] == "table":
            cur = {"params": tuple(int(v) for v in ln[1:]), "rows": []}
            out.append(cur)
        else:
            cur["rows"].append([int(v) for v in ln])
    return out


def test_triton_tables():
    tabs = _triton_tables()
    assert len(tabs) == 5
    for t in tabs:
        vec, per_phase, max_phase, rows, cols = t["params"]
        assert sb.triton_table(rows, cols, vec, per_phase, max_phase) == t["rows"], t["params"]


def _fixture():
    return {ln[0]: int(ln[1]) for ln in read_lines("sbc_transpose_conflicts.txt")
            if ln[0] != "M"}


def test_transpose_conflict_counts():
    g = _fixture()
    st, ld = sb.transpose_conflict_totals("naive", 1024, 2048)
    assert st == g["naive_store_conflicts"]
    assert ld == 0
    # wavefronts: one per conflict plus one per warp store
    warp_stores = (1024 * 2048) // 32
    assert st + warp_stores == g["naive_store_wavefronts"]
    assert sb.transpose_conflict_totals("padded", 1024, 2048) == (g["padded_store_conflicts"], 0)
    assert sb.transpose_conflict_totals("xor", 1024, 2048) == (g["xor_store_conflicts"], 0)


def test_transpose_conflicts_large_closed_form():
    # every warp store of the naive layout hits one bank 32 times: 31 extra
    st, _ = sb.transpose_conflict_totals("naive", 16384, 32768)
    assert st == (16384 * 32768 // 32) * 31 == 520093696


def test_wavefront_rules():
    # 32 lanes reading 32 consecutive words: 1 wavefront
    assert sb.wavefronts([4 * t for t in range(32)], 4) == 1
    # all lanes reading the same word: broadcast, 1 wavefront
    assert sb.wavefronts([0] * 32, 4) == 1
    # stride 2 words: 2-way conflict
    assert sb.wavefronts([8 * t for t in range(32)], 4) == 2
    # 16-byte accesses: 4 phases of 8 lanes, contiguous -> 4 wavefronts, 0 conflicts
    assert sb.wavefronts([16 * t for t in range(32)], 16) == 4
    assert sb.conflicts([16 * t for t in range(32)], 16) == 0
    # 8-byte accesses: 2 phases
    assert sb.wavefronts([8 * t for t in range(32)], 8) == 2


@pytest.mark.parametrize("fn", ["xor", "tma"])
def test_swizzle_properties(fn):
    """The page's three properties of a swizzle map: one-to-one, ranges kept,
    and two rows never put the same logical column in the same physical one."""
    rows, cols = (32, 32) if fn == "xor" else (8, 64)

    def phys(r, c):
        if fn == "xor":
            return r, sb.xor_offset(r, c, cols) - r * cols
        return sb.tma_swizzle_128b(r, c, cols, 2)

    images = {phys(r, c) for r in range(rows) for c in range(cols)}
    assert len(images) == rows * cols
    assert all(0 <= y < rows and 0 <= x < cols for y, x in images)
    for c in range(cols):
        xs = [phys(r, c)[1] for r in range(rows)]
        if fn == "xor":
            assert len(set(xs)) == rows
        else:  # chunk granularity: 8 rows of one atom land in 8 distinct chunks
            assert len({x // 8 for x in xs}) == rows


def test_tma_swizzle_equals_cute_swizzle():
    # Swizzle<3,3,3> on fp16 element offsets and Swizzle<3,4,3> on byte
    # offsets describe the same 128-byte swizzle as the TMA chunk formula.
    for y in range(16):
        for x in range(64):
            yy, xs = sb.tma_swizzle_128b(y, x, 64, 2)
            assert yy * 64 + xs == sb.cute_swizzle(y * 64 + x, 3, 3, 3)
            assert 2 * (yy * 64 + xs) == sb.cute_swizzle(2 * (y * 64 + x), 3, 4, 3)
    # 4-byte elements: 32 per 128-byte row, chunk = 4 elements
    for y in range(8):
        for x in range(32):
            yy, xs = sb.tma_swizzle_128b(y, x, 32, 4)
            assert 4 * (yy * 32 + xs) == sb.cute_swizzle(4 * (y * 32 + x), 3, 4, 3)


def test_staged_epilogue_store_conflicts():
    # 128-byte rows, lane t writes 16 bytes of row t: without the swizzle the
    # 8 lanes of a phase hit the same 4 banks (8 wavefronts per phase, 28
    # extra over the 4 phases); with it every phase is conflict free.
    assert sb.staged_row_store_conflicts(128, swizzled=False) == [28] * 8
    assert sb.staged_row_store_conflicts(128, swizzled=True) == [0] * 8


def test_padding_breaks_16b_alignment():
    # the page's caveat: in int[32][33], row 1 starts at byte 132, not 16-aligned
    assert (sb.padded_offset(1, 0, 32) * 4) % 16 != 0


def test_ldmatrix_conflict_model():
    # Rows 128 bytes apart (64 fp16 elements) share one bank group: the 8
    # lanes of an ldmatrix phase that name 8 consecutive rows at one column
    # chunk serialise 8-fold -> 7 extra wavefronts per phase, 28 per x4.
    naive, pad, swz128, swz64 = (8, 1, 1, 0), (8, 1, 1, 8), (8, 1, 8, 0), (8, 2, 4, 0)
    assert sb.conflicts(sb.ldmatrix_x4_addresses(0, 0, 64, naive), 16) == 28
    assert sb.conflicts(sb.ldmatrix_x4_addresses(0, 0, 128, naive), 16) == 28
    # 16 bytes of padding shift each row by 4 banks: conflict free
    assert sb.conflicts(sb.ldmatrix_x4_addresses(16, 8, 64, pad), 16) == 0
    # chunk XOR row (mod 8) puts the 8 rows of a phase into 8 bank groups
    for r0, c0 in [(0, 0), (16, 16), (48, 48)]:
        assert sb.conflicts(sb.ldmatrix_x4_addresses(r0, c0, 64, swz128), 16) == 0
    # two rows per phase value: pairs of rows collide -> 2-way, 4 per x4
    assert sb.conflicts(sb.ldmatrix_x4_addresses(0, 0, 64, swz64), 16) == 4
    # the Swizzle<3,3,3> formula of the CUTLASS section equals the (8,1,8)
    # Triton layout on 64-element rows
    for r in range(16):
        for c in range(64):
            assert sb.staged_offset(r, c, 64, *swz128) == sb.cute_swizzle(r * 64 + c, 3, 3, 3)


def test_mma_sync_kernel_conflict_totals():
    # per CTA and 64-deep K block (8 warps x 4 steps x 6 ldmatrix.x4)
    lays = {"naive": (8, 1, 1, 0), "padded": (8, 1, 1, 8), "swz128": (8, 1, 8, 0),
            "swz64": (8, 2, 4, 0)}
    want = {"naive": 8 * 4 * 6 * 28, "padded": 0, "swz128": 0, "swz64": 8 * 4 * 6 * 4}
    for name, lay in lays.items():
        got = sum(sb.ldmatrix_conflicts_per_k_step(lay, lay, wm * 64, wn * 32, ks * 16, 64, 128)
                  for wm in range(2) for wn in range(4) for ks in range(4))
        assert got == want[name], name
        assert sb.cp_async_tile_conflicts(128, 64, lay) == 0
        assert sb.cp_async_tile_conflicts(64, 128, lay) == 0


def test_tma_swizzle_spans_pinned():
    # 128-byte span: the page's chunk formula on 128-byte rows
    for y in range(16):
        for x in range(64):
            yy, xs = sb.tma_swizzle_128b(y, x, 64, 2)
            assert sb.tma_swizzle_bytes(2 * (y * 64 + x), 128) == 2 * (yy * 64 + xs)
    # every span: Swizzle<b,4,3> of the CUTLASS section on byte addresses
    for span, b in ((128, 3), (64, 2), (32, 1)):
        for a in range(0, 4096, 2):
            assert sb.tma_swizzle_bytes(a, span) == sb.cute_swizzle(a, b, 4, 3)
    # 64- and 32-byte spans as Triton layouts on rows of 32 / 16 fp16
    # elements: (vec 8, perPhase 2, maxPhase 4) and (vec 8, perPhase 4,
    # maxPhase 2) -- the stored column of each chunk matches
    for span, pp, mp in ((64, 2, 4), (32, 4, 2)):
        w = span // 2
        for r in range(16):
            for c in range(w):
                phys = sb.tma_swizzle_bytes(2 * (r * w + c), span) // 2 - r * w
                assert sb.triton_source_column(r, phys, 8, pp, mp) == c


@pytest.mark.parametrize("span", [128, 64, 32])
def test_tma_swizzle_permutes_chunks(span):
    block = 8 * span
    for base in (0, block, 5 * block):
        img = [sb.tma_swizzle_bytes(base + a, span) for a in range(0, block, 16)]
        assert sorted(img) == list(range(base, base + block, 16))  # chunks permuted in place
        assert all(sb.tma_swizzle_bytes(base + a + 4, span) == i + 4
                   for a, i in zip(range(0, block, 16), img))   # bytes stay in their chunk


@pytest.mark.parametrize("span", [128, 64, 32])
def test_core_matrix_reads_conflict_free(span):
    # 8 rows x 16 bytes at every 16-byte position of the row: one wavefront
    # with the swizzle; without it, rows `span` bytes apart collide: span / 16
    # of the 8 rows share each 16-byte bank group
    for k in range(0, span, 16):
        addrs = sb.core_matrix_read_addresses(8, k, span)
        assert sb.wavefronts(addrs, 16) == 1
        plain = sb.core_matrix_read_addresses(8, k, span, swizzled=False)
        assert sb.wavefronts(plain, 16) == span // 16
