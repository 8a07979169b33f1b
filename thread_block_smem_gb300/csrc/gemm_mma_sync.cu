// gemm_mma_sync.cu -- C = A * B on the warp-level tensor-core path
// (cp.async -> shared memory -> ldmatrix -> mma.sync.m16n8k16), with the
// shared-memory layout of the operand tiles chosen at run time.
//
// Purpose: the operand swizzle of the main GEMM is read by the tensor core
// itself and cannot be observed with load/store-unit counters; this kernel
// loads every fragment with ldmatrix through the load/store unit, so the
// bank conflicts a layout causes are visible (and countable) -- the
// situation of WHC, "CUDA Swizzle & bank conflict", section "MMA Bank
// Conflict" (ldmatrix in four 8-lane phases, each lane naming one 16-byte
// row; rows one 128-byte line apart hit the same banks).
//
// Layouts (element (r, c) of a tile with rows of W elements):
//   offset = r * (W + pad) + ((c / vec) ^ ((r / per_phase) % max_phase)) * vec + c % vec
// the shared layout of "Triton - Shared Layout swizzling" (vec, perPhase,
// maxPhase) plus optional padding ("Padding"); max_phase = 1, pad = 0 is the
// plain row-major tile; vec = 8, per_phase = 1, max_phase = 8 on 64-element
// fp16 rows is Swizzle<3,3,3> of "swizzle in CUTLASS".
//
// CTA tile 128 x 128 x 64, 256 threads = 8 warps as 2 (M) x 4 (N), warp tile
// 64 x 32; two cp.async stages; one CTA per output tile, tile = order(id).
#include "common.h"
#include "tile_order.cuh"

namespace swz {
namespace mmasync {

constexpr int BM = 128, BN = 128, BK = 64;

struct Layout {
  int vec, per_phase, max_phase, pad;
};

struct Params {
  const uint16_t* A;
  const uint16_t* B;
  float* C;
  int M, N, K;
  int order, group;
  uint32_t gm, gn;
  Layout la, lb;
};

__device__ __forceinline__ uint32_t tile_elem(const Layout& L, int width, int r, int c) {
  const int phase = (r / L.per_phase) % L.max_phase;
  return uint32_t(r * (width + L.pad) + ((c / L.vec) ^ phase) * L.vec + c % L.vec);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool BF16>
__global__ void __launch_bounds__(256) mma_sync_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int a_elems = BM * (BK + p.la.pad), b_elems = BK * (BN + p.lb.pad);
  const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  auto sA = [&](int st) { return s0 + uint32_t(st * (a_elems + b_elems) * 2); };
  auto sB = [&](int st) { return sA(st) + uint32_t(a_elems * 2); };

  const TileCoord t = tile_of(p.order, blockIdx.x, p.gm, p.gn, uint32_t(p.group));
  const int m0 = int(t.m) * BM, n0 = int(t.n) * BN;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int wm = (warp / 4) * 64, wn = (warp % 4) * 32;
  const int nkb = (p.K + BK - 1) / BK;

  // 16-byte chunks: A tile 128 rows x 8 chunks, B tile 64 rows x 16 chunks;
  // thread tid copies chunks tid, tid + 256, tid + 512, tid + 768 of each
  auto load = [&](int st, int kb) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ca = tid + 256 * j;
      const int ra = ca / 8, ka = (ca % 8) * 8;
      const int gr = m0 + ra, gk = kb * BK + ka;
      const bool va = gr < p.M && gk < p.K;
      cp_async16(sA(st) + 2 * tile_elem(p.la, BK, ra, ka),
                 p.A + (va ? size_t(gr) * p.K + gk : 0), va);
      const int rb = ca / 16, nb = (ca % 16) * 8;
      const int gkb = kb * BK + rb, gn = n0 + nb;
      const bool vb = gkb < p.K && gn < p.N;
      cp_async16(sB(st) + 2 * tile_elem(p.lb, BN, rb, nb),
                 p.B + (vb ? size_t(gkb) * p.N + gn : 0), vb);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[i][j][v] = 0.f;

  load(0, 0);
  for (int kb = 0; kb < nkb; ++kb) {
    const int st = kb & 1;
    if (kb + 1 < nkb) {
      load(st ^ 1, kb + 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int q = lane / 8, i8 = lane % 8;
#pragma unroll
    for (int ks = 0; ks < BK; ks += 16) {
      uint32_t af[4][4], bf[2][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        ldsm_x4(sA(st) + 2 * tile_elem(p.la, BK, wm + 16 * mt + i8 + 8 * (q % 2), ks + 8 * (q / 2)),
                af[mt]);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        ldsm_x4_trans(
            sB(st) + 2 * tile_elem(p.lb, BN, ks + i8 + 8 * (q % 2), wn + 16 * nt + 8 * (q / 2)),
            bf[nt]);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          mma16816<BF16>(acc[mt][nt], af[mt], bf[nt / 2][2 * (nt % 2)],
                         bf[nt / 2][2 * (nt % 2) + 1]);
    }
    __syncthreads();
  }

  // fragment layout of D: rows lane/4 and lane/4 + 8, columns 2*(lane%4) + {0,1}
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = m0 + wm + 16 * mt + lane / 4 + 8 * h;
        const int c = n0 + wn + 8 * nt + 2 * (lane % 4);
        if (r < p.M && c < p.N)
          *reinterpret_cast<float2*>(p.C + size_t(r) * p.N + c) =
              make_float2(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
      }
}

bool layout_ok(const Layout& L, int width) {
  auto pow2 = [](int x) { return x > 0 && (x & (x - 1)) == 0; };
  if (!pow2(L.vec) || L.vec % 8 || !pow2(L.per_phase) || !pow2(L.max_phase)) return false;
  if (L.max_phase * L.vec > width) return false;  // XOR stays inside the row
  if (L.pad < 0 || L.pad % 8 || L.pad > 64) return false;
  return true;
}

}  // namespace mmasync
}  // namespace swz

using namespace swz;
using namespace swz::mmasync;

extern "C" int swz_gemm_mma_sync(const void* A, const void* B, float* C, int M, int N, int K,
                                 int dtype, int vec, int per_phase, int max_phase, int pad,
                                 int order, int group, void* stream) {
  if (M < 0 || N < 0 || K < 0 || (dtype != SWZ_F16 && dtype != SWZ_BF16)) return SWZ_EINVAL;
  if (!order_is_valid(order) || (order_uses_group(order) && group < 1)) return SWZ_EINVAL;
  const Layout L{vec, per_phase, max_phase, pad};
  if (!layout_ok(L, BK) || !layout_ok(L, BN)) return SWZ_EINVAL;
  if (M == 0 || N == 0) return SWZ_OK;
  if (!C || (reinterpret_cast<uintptr_t>(C) & 7u)) return SWZ_EINVAL;
  if (K > 0 && (!A || !B || !aligned16(A) || !aligned16(B))) return SWZ_EINVAL;
  if (K % 8 || N % 8) return SWZ_EINVAL;
  DeviceInfo dev{};
  int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    SWZ_CUDA_TRY(cudaMemsetAsync(C, 0, size_t(M) * N * sizeof(float), s));
    return SWZ_OK;
  }
  const uint32_t gm = uint32_t((M + BM - 1) / BM), gn = uint32_t((N + BN - 1) / BN);
  if (uint64_t(gm) * gn > uint64_t(INT32_MAX)) return SWZ_EINVAL;
  const uint32_t g = order_uses_group(order) ? uint32_t(group) : 1u;
  if ((order == kMorton || order == kXor) && !order_is_bijective(order, gm, gn, g))
    return SWZ_ENOTBIJECTIVE;
  Params prm{};
  prm.A = static_cast<const uint16_t*>(A);
  prm.B = static_cast<const uint16_t*>(B);
  prm.C = C;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.order = order;
  prm.group = int(g);
  prm.gm = gm;
  prm.gn = gn;
  prm.la = L;
  prm.lb = L;
  const size_t smem = 2 * (size_t(BM) * (BK + pad) + size_t(BK) * (BN + pad)) * 2;
  if (dtype == SWZ_BF16) {
    SWZ_CUDA_TRY(cudaFuncSetAttribute(mma_sync_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    mma_sync_kernel<true><<<gm * gn, 256, smem, s>>>(prm);
  } else {
    SWZ_CUDA_TRY(cudaFuncSetAttribute(mma_sync_kernel<false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
    mma_sync_kernel<false><<<gm * gn, 256, smem, s>>>(prm);
  }
  SWZ_CUDA_TRY(cudaGetLastError());
  return SWZ_OK;
}
