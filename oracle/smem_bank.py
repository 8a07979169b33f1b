"""Shared-memory address functions and a bank-conflict counter (oracle).

Source: WHC, "CUDA Swizzle & bank conflict":
  * "Bank" / "Bank Conflict": 32 banks of 4 bytes; threads of one phase that
    touch different 4-byte words of one bank are serialised, identical words
    are broadcast.
  * "memory coalesce": 128-bit accesses run in 4 phases of 8 threads (16-byte
    units, 8 "virtual banks"); 64-bit accesses in 2 phases of 16 threads.
  * "Padding" ([32][33] and r*(cols+1)+c), "swizzle 原理" (the three properties
    of a swizzle map), "Matrix Transpose" (naive / padded / XOR-swizzled tiles
    and the conflict and wavefront arithmetic), "Hopper TMA 的 swizzling" (the
    128-byte chunk formula), "swizzle in CUTLASS" (Swizzle<B,M,S>) and
    "Triton - Shared Layout swizzling" (vec / perPhase / maxPhase).

Addresses here are plain integers (element or byte offsets from the start of
the shared array); nothing touches a GPU.
"""
from __future__ import annotations

NUM_BANKS = 32
BANK_BYTES = 4


# ----------------------------------------------------------------------------
# address functions
# ----------------------------------------------------------------------------
def naive_offset(r, c, cols):
    """Row-major element offset of (r, c) in a rows x cols array."""
    return r * cols + c


def padded_offset(r, c, cols):
    """Row-major offset in a rows x (cols+1) array: each row shifted by one
    element, i.e. one bank for 4-byte elements ("Padding")."""
    return r * (cols + 1) + c


def xor_offset(r, c, cols):
    """Element offset of logical (r, c) when the column is XOR-ed with the row
    ("Matrix Transpose", swizzling kernel: physical column = c ^ r).  cols
    must be a power of two no smaller than the row count."""
    return r * cols + (c ^ r)


def tma_swizzle_128b(y, x, nx, elem_bytes):
    """Physical (y, x) of logical element [y][x] of ``T array[][nx]`` under the
    128-byte TMA swizzle ("Hopper TMA 的 swizzling"): 16-byte chunks are
    numbered i16 = (y*nx + x)*sizeof(T)/16, split into a chunk row i16 div 8
    and a chunk column i16 mod 8; the chunk column is XOR-ed with the chunk
    row; the element keeps its place inside its chunk.  Requires
    nx * sizeof(T) == 128."""
    if nx * elem_bytes != 128:
        raise ValueError("128B swizzle needs rows of exactly 128 bytes")
    per_chunk = 16 // elem_bytes
    i16 = (y * nx + x) * elem_bytes // 16
    y16, x16 = i16 // 8, i16 % 8
    x16_swz = y16 ^ x16
    x_swz = (x16_swz * per_chunk) % nx + x % per_chunk
    return y, x_swz


def cute_swizzle(offset, b, m, s):
    """Swizzle<B,M,S> ("swizzle in CUTLASS"): units of 2^M are never split;
    the B bits just above them (bits [M, M+B)) are XOR-ed with the B bits that
    sit S positions higher (bits [M+S, M+S+B))."""
    mask = ((1 << b) - 1) << (m + s)
    return offset ^ ((offset & mask) >> s)


def tma_swizzle_bytes(addr, span):
    """Physical byte address of logical byte address ``addr`` (relative to a
    base aligned to the pattern) under the TMA / tensor-core swizzle of span
    ``span`` = 128, 64 or 32 bytes.  Generalises the 128-byte rule of "Hopper
    TMA 的 swizzling" as the PTX ISA's swizzle modes state it: the 16-byte
    chunk bits of the address (bits 4 ..) are XOR-ed with the same number of
    bits of the 128-byte line index (bits 7 ..); the span fixes how many:
    3 for 128 bytes, 2 for 64, 1 for 32.  The pattern repeats every
    8 * span bytes."""
    bits = {128: 3, 64: 2, 32: 1}[span]
    mask = (1 << bits) - 1
    return addr ^ (((addr >> 7) & mask) << 4)


def core_matrix_read_addresses(rows, k_byte, span, swizzled=True):
    """Byte addresses of one 16-byte read from each of ``rows`` consecutive
    rows of a K-major operand block whose rows are ``span`` bytes long (one
    swizzle column group), at byte ``k_byte`` of the row: the pattern of a
    tensor-core core-matrix read (8 rows x 16 bytes)."""
    out = []
    for r in range(rows):
        a = r * span + k_byte
        out.append(tma_swizzle_bytes(a, span) if swizzled else a)
    return out


def triton_source_column(r, c, vec, per_phase, max_phase):
    """Triton shared layout ("Triton - Shared Layout swizzling"): element
    (r, c) of the stored tile holds input column
    ((c div vec) XOR ((r div perPhase) mod maxPhase)) * vec + c mod vec."""
    phase = (r // per_phase) % max_phase
    return ((c // vec) ^ phase) * vec + c % vec


def triton_table(rows, cols, vec, per_phase, max_phase):
    """The stored tile for input [0, 1, ..., rows*cols-1] (row-major)."""
    return [[r * cols + triton_source_column(r, c, vec, per_phase, max_phase)
             for c in range(cols)] for r in range(rows)]


# ----------------------------------------------------------------------------
# bank-conflict counting
# ----------------------------------------------------------------------------
def wavefronts(byte_addrs, width_bytes):
    """Wavefronts one warp-wide shared access needs.

    ``byte_addrs[t]`` is the start address of lane t (None = inactive);
    ``width_bytes`` is 4, 8 or 16.  Lanes are split into phases of
    32*4/width lanes; inside a phase, the cost is the largest number of
    distinct 4-byte words that fall into one bank (at least 1 if any lane is
    active)."""
    lanes_per_phase = NUM_BANKS * BANK_BYTES // width_bytes
    total = 0
    for p0 in range(0, len(byte_addrs), lanes_per_phase):
        words_by_bank = {}
        for a in byte_addrs[p0:p0 + lanes_per_phase]:
            if a is None:
                continue
            if a % width_bytes:
                raise ValueError("misaligned shared access")
            for w in range(a // BANK_BYTES, (a + width_bytes) // BANK_BYTES):
                words_by_bank.setdefault(w % NUM_BANKS, set()).add(w)
        if words_by_bank:
            total += max(len(v) for v in words_by_bank.values())
    return total


def ideal_wavefronts(byte_addrs, width_bytes):
    lanes_per_phase = NUM_BANKS * BANK_BYTES // width_bytes
    return sum(1 for p0 in range(0, len(byte_addrs), lanes_per_phase)
               if any(a is not None for a in byte_addrs[p0:p0 + lanes_per_phase]))


def conflicts(byte_addrs, width_bytes):
    """Extra wavefronts beyond one per active phase."""
    return wavefronts(byte_addrs, width_bytes) - ideal_wavefronts(byte_addrs, width_bytes)


_LAYOUTS = {"naive": naive_offset, "padded": padded_offset, "xor": xor_offset}


def transpose_tile_accesses(layout, ty, tile=32, elem_bytes=4):
    """Byte addresses of the two shared accesses of warp ``ty`` in the 32x32
    transpose ("Matrix Transpose"): lane tx stores the element it loaded from
    global (row ty, column tx) at logical [tx][ty], then reads logical
    [ty][tx] for the coalesced global store."""
    off = _LAYOUTS[layout]
    store = [off(tx, ty, tile) * elem_bytes for tx in range(tile)]
    load = [off(ty, tx, tile) * elem_bytes for tx in range(tile)]
    return store, load


def transpose_conflict_totals(layout, M, N, tile=32):
    """Total (store, load) bank conflicts of the shared-memory transpose of an
    M x N matrix of 4-byte words: every 32x32 tile runs 32 warp stores and 32
    warp loads, one per tile row."""
    st = ld = 0
    for ty in range(tile):
        s, l_ = transpose_tile_accesses(layout, ty, tile)
        st += conflicts(s, 4)
        ld += conflicts(l_, 4)
    tiles = (M // tile) * (N // tile)
    return st * tiles, ld * tiles


def staged_row_store_conflicts(row_bytes, swizzled):
    """Conflicts of one warp-wide 16-byte store into a staging tile whose
    rows are ``row_bytes`` long, lane t writing chunk j of row t, for every
    chunk index j of the row.  With ``swizzled`` the chunk is placed at
    j XOR (t mod 8) (the 128-byte TMA swizzle applied to a 128-byte row).
    Returns the list of conflicts per j."""
    chunks = row_bytes // 16
    out = []
    for j in range(chunks):
        addrs = []
        for t in range(32):
            jj = (j ^ (t % 8)) % chunks if swizzled else j
            addrs.append(t * row_bytes + jj * 16)
        out.append(conflicts(addrs, 16))
    return out


# ----------------------------------------------------------------------------
# ldmatrix / cp.async operand staging ("MMA Bank Conflict", "swizzle in
# CUTLASS", "Triton - Shared Layout swizzling")
# ----------------------------------------------------------------------------
def staged_offset(r, c, width, vec, per_phase, max_phase, pad):
    """Element offset of logical (r, c) in a tile with rows of `width`
    elements plus `pad` elements of padding, under the Triton-style swizzle
    (vec, perPhase, maxPhase); max_phase = 1 is the plain row-major tile."""
    return r * (width + pad) + triton_source_column(r, c, vec, per_phase, max_phase)


def ldmatrix_x4_addresses(r0, c0, width, layout, elem_bytes=2, trans_b=False):
    """Byte addresses the 32 lanes of one ldmatrix.x4 supply for the 16 x 16
    block at (r0, c0): lane l names row (l mod 8) of 8 x 8 matrix l div 8.
    For the A operand (row-major M x K tile) matrix q covers rows
    r0 + 8*(q mod 2) and columns c0 + 8*(q div 2); for the B operand loaded
    with .trans (K x N tile, N contiguous) matrix q covers k rows
    r0 + 8*(q mod 2) and n columns c0 + 8*(q div 2) as well."""
    vec, per_phase, max_phase, pad = layout
    out = []
    for lane in range(32):
        q, i = lane // 8, lane % 8
        r = r0 + i + 8 * (q % 2)
        c = c0 + 8 * (q // 2)
        out.append(staged_offset(r, c, width, vec, per_phase, max_phase, pad) * elem_bytes)
    return out


def ldmatrix_conflicts_per_k_step(layout_a, layout_b, warp_m0, warp_n0, bk_step,
                                  width_a, width_b):
    """Bank conflicts of one warp's fragment loads for one 16-deep K step of
    the mma.sync GEMM: four ldmatrix.x4 over A rows warp_m0 .. +63 and two
    ldmatrix.x4.trans over B columns warp_n0 .. +31."""
    total = 0
    for mt in range(4):
        total += conflicts(ldmatrix_x4_addresses(warp_m0 + 16 * mt, bk_step, width_a,
                                                 layout_a), 16)
    for nt in range(2):
        total += conflicts(ldmatrix_x4_addresses(bk_step, warp_n0 + 16 * nt, width_b,
                                                 layout_b), 16)
    return total


def cp_async_tile_conflicts(rows, width, layout, threads=256):
    """Bank conflicts of the 16-byte cp.async writes that fill one tile of
    `rows` x `width` halves: chunk t (row t div (width/8), 8-element column
    group t mod (width/8)) is written by thread t mod threads; each warp
    instruction writes 32 consecutive chunks."""
    per_row = width // 8
    chunks = rows * per_row
    total = 0
    for base in range(0, chunks, 32):
        addrs = []
        for t in range(base, min(base + 32, chunks)):
            r, g = divmod(t, per_row)
            addrs.append(staged_offset(r, 8 * g, width, *layout) * 2)
        total += conflicts(addrs, 16)
    return total
