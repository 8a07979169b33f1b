// transpose.cu -- shared-memory-staged transpose of 32-bit words with the
// three tile layouts of WHC, "CUDA Swizzle & bank conflict", section "Matrix
// Transpose": naive tile[32][32], padded tile[32][33] and XOR-swizzled
// tile[32][32] whose element (r, c) sits in column c ^ r.
//
// Per 32 x 32 tile: lane tx of warp ty loads input row
// (r0 + ty + 8i), column (c0 + tx) -- a coalesced 128-byte row segment -- and
// stores it at logical tile[tx][ty + 8i]; after the barrier it reads logical
// tile[ty + 8i][tx] and writes output row (c0 + ty + 8i), column (r0 + tx),
// again 128 contiguous bytes per warp.  The store phase is where the layouts
// differ: with the naive layout the 32 lanes of a warp write 32 different
// rows of one tile column, all in one bank (31 extra wavefronts per warp
// store); the padded and XOR layouts spread them over all 32 banks.
//
// Differences from the page's kernel: 256 threads per CTA (32 x 8), each CTA
// moving four 32 x 32 tiles that sit side by side along N, with four rows
// per thread and tile, so that 16 loads are in flight per thread (the
// one-tile form reached 78 % of the copy bandwidth, four tiles 99 %); the
// barrier sits outside any bounds test, so ragged M and N are handled by
// clipping the global accesses.  The warp-level shared-memory access pattern
// -- and so the conflict count per warp store -- is the page's.
#include "common.h"

namespace swz {

template <int LAYOUT>
__device__ __forceinline__ int tile_offset(int r, int c) {
  if constexpr (LAYOUT == SWZ_SMEM_NAIVE) return r * 32 + c;
  if constexpr (LAYOUT == SWZ_SMEM_PADDED) return r * 33 + c;
  return r * 32 + (c ^ r);
}

constexpr int kTilesPerCta = 4;  // 32 x 32 tiles side by side along N

template <int LAYOUT>
__global__ void __launch_bounds__(256) transpose_kernel(const uint32_t* __restrict__ in,
                                                        uint32_t* __restrict__ out, int M, int N) {
  __shared__ uint32_t tile[kTilesPerCta][32 * 33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t r0 = int64_t(blockIdx.y) * 32;
  const int64_t cb = int64_t(blockIdx.x) * 32 * kTilesPerCta;
  // all loads first: 16 independent 4-byte loads per thread in flight
  uint32_t v[kTilesPerCta][4];
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t gr = r0 + ty + 8 * i, gc = cb + 32 * t + tx;
      v[t][i] = (gr < M && gc < N) ? __ldg(in + gr * N + gc) : 0u;
    }
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) tile[t][tile_offset<LAYOUT>(tx, ty + 8 * i)] = v[t][i];
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty + 8 * i;
      const int64_t orow = cb + 32 * t + r, ocol = r0 + tx;
      if (orow < N && ocol < M) out[orow * M + ocol] = tile[t][tile_offset<LAYOUT>(r, tx)];
    }
}

}  // namespace swz

using namespace swz;

extern "C" int swz_transpose(const uint32_t* in, uint32_t* out, int M, int N, int layout,
                             void* stream) {
  if (M < 0 || N < 0) return SWZ_EINVAL;
  if (layout < SWZ_SMEM_NAIVE || layout > SWZ_SMEM_XOR) return SWZ_EINVAL;
  if (M == 0 || N == 0) return SWZ_OK;
  if (!in || !out || !aligned4(in) || !aligned4(out)) return SWZ_EINVAL;
  const int64_t tiles_m = (int64_t(M) + 31) / 32;
  const int64_t tiles_n = (int64_t(N) + 32 * kTilesPerCta - 1) / (32 * kTilesPerCta);
  if (tiles_m > 65535) return SWZ_EINVAL;
  const uint64_t bytes = uint64_t(M) * uint64_t(N) * 4u;
  const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
  if (a < b + bytes && b < a + bytes) return SWZ_EINVAL;  // overlapping buffers
  DeviceInfo dev{};
  const int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  const dim3 grid{static_cast<unsigned>(tiles_n), static_cast<unsigned>(tiles_m), 1u};
  const dim3 block{32u, 8u, 1u};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (layout) {
    case SWZ_SMEM_NAIVE: transpose_kernel<SWZ_SMEM_NAIVE><<<grid, block, 0, s>>>(in, out, M, N); break;
    case SWZ_SMEM_PADDED: transpose_kernel<SWZ_SMEM_PADDED><<<grid, block, 0, s>>>(in, out, M, N); break;
    default: transpose_kernel<SWZ_SMEM_XOR><<<grid, block, 0, s>>>(in, out, M, N); break;
  }
  SWZ_CUDA_TRY(cudaGetLastError());
  return SWZ_OK;
}
