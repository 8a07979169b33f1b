// tile_order.cuh -- program-id -> output-tile maps and the persistent
// work-index stride, usable on host and device.
//
// Orders (ids as in include/swz.h):
//   row / col-major, grouped 2D panel, Morton, XOR: Lei Mao, "CUDA Thread
//     Block Swizzle", sections "Linear Swizzle", "Grouped 2D Panel Swizzle",
//     "Morton / Z-order Swizzle", "Bitwise XOR Swizzle" and the benchmark's
//     device mapping function.
//   serpentine: TVM TIRx "ClusterPersistentScheduler2D", section "Serpentine
//     Mode", read from its 4x4 example table: column strips S tiles wide,
//     rows of a strip walked downwards in even strips and upwards in odd ones,
//     left to right inside a row; a narrower last strip uses its own width.
//   group-major ("Tile Ordering" on the same page) is the panel order.
//
// All arithmetic is 32-bit unsigned on non-negative ids: id < gm*gn < 2^31.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SWZ_HD __host__ __device__ __forceinline__
#else
#define SWZ_HD inline
#endif

namespace swz {

enum Order : int { kRow = 0, kCol = 1, kPanel = 2, kMorton = 3, kXor = 4, kSerpentine = 5 };

struct TileCoord {
  uint32_t m, n;
};

// Grouped panel: bands of `g` tile rows; ids run down the band's columns.
SWZ_HD TileCoord panel_tile(uint32_t id, uint32_t gm, uint32_t gn, uint32_t g) {
  const uint32_t band_size = g * gn;
  const uint32_t band = id / band_size;
  const uint32_t row0 = band * g;
  const uint32_t rows = (gm - row0 < g) ? gm - row0 : g;
  const uint32_t r = id - band * band_size;
  return {row0 + r % rows, r / rows};
}

// Morton: even bits of id form m, odd bits form n (compacted with the
// classic mask-and-shift sequence), reduced modulo the grid.
SWZ_HD uint32_t compact_even_bits(uint32_t x) {
  x &= 0x55555555u;
  x = (x | (x >> 1)) & 0x33333333u;
  x = (x | (x >> 2)) & 0x0F0F0F0Fu;
  x = (x | (x >> 4)) & 0x00FF00FFu;
  x = (x | (x >> 8)) & 0x0000FFFFu;
  return x;
}

SWZ_HD TileCoord morton_tile(uint32_t id, uint32_t gm, uint32_t gn) {
  return {compact_even_bits(id) % gm, compact_even_bits(id >> 1) % gn};
}

SWZ_HD TileCoord xor_tile(uint32_t id, uint32_t gm, uint32_t gn) {
  const uint32_t y = id / gn;
  const uint32_t x = id - y * gn;
  return {(x ^ y) % gm, y % gn};
}

SWZ_HD TileCoord serpentine_tile(uint32_t id, uint32_t gm, uint32_t gn, uint32_t s) {
  const uint32_t strip_size = s * gm;
  const uint32_t strip = id / strip_size;
  const uint32_t r = id - strip * strip_size;
  const uint32_t n0 = strip * s;
  const uint32_t width = (gn - n0 < s) ? gn - n0 : s;
  const uint32_t step = r / width;
  const uint32_t m = (strip & 1u) ? gm - 1u - step : step;
  return {m, n0 + (r - step * width)};
}

SWZ_HD TileCoord tile_of(int order, uint32_t id, uint32_t gm, uint32_t gn, uint32_t group) {
  switch (order) {
    case kRow: return {id / gn, id % gn};
    case kCol: return {id % gm, id / gm};
    case kPanel: return panel_tile(id, gm, gn, group);
    case kMorton: return morton_tile(id, gm, gn);
    case kXor: return xor_tile(id, gm, gn);
    default: return serpentine_tile(id, gm, gn, group);
  }
}

SWZ_HD bool order_is_valid(int order) { return order >= kRow && order <= kSerpentine; }
SWZ_HD bool order_uses_group(int order) { return order == kPanel || order == kSerpentine; }

}  // namespace swz
