// tc_rate.cu -- swz_tc_rate: how many FLOP per SM clock the tcgen05 tensor
// cores retire, measured with this library's own MMA code.
//
// The GEMM's roofline needs a dense tensor peak.  Instead of taking a figure
// from a data sheet, this kernel keeps every SM's tensor core busy with
// back-to-back tcgen05.mma instructions whose operands sit in shared memory
// (no memory traffic at all) and times them with the SM's cycle counter and
// the global nanosecond timer.  FLOP per clock per SM follows from the
// instruction count; peak = SMs x that x SM clock, at the maximum clock or
// at the clock the run itself saw (the ratio cycles / ns).
//
// Design: one CTA per SM (the shared-memory request leaves room for one);
// 4 warps.  All threads copy the caller's A (128 x 128 bytes) and B
// (n x 128 bytes, K-major; with a CTA pair each CTA takes its half of B's
// rows) into the 128-byte-swizzled layout the GEMM uses; warp 0 allocates
// 256 TMEM columns; thread 0 (of the pair's leader) issues n_mma MMAs of
// shape 128 x n x k (256 x n x k for a pair; k = 16 for fp16/bf16, 8 for
// TF32) cycling through the four k-slices of the 128-byte rows, all into
// one fp32 accumulator, commits, waits (bounded) and records its cycle and
// time spans.  CTA 0 then copies the accumulator out so a caller can check
// the MMAs really ran: with n_mma a multiple of 4 it holds
// (n_mma / 4) * A * B^T.
//
// Stage mode (S MMAs per stage): the issue loop is cut into stages the way
// the GEMM's is -- per stage one non-blocking test of a barrier (one whose
// phase is already complete, so no wait ever happens), the tensor fence, S
// MMAs and a commit to a second barrier -- unrolled by 8.  It measures what
// the issuing thread's per-stage work costs the tensor pipe, with the
// operands already in shared memory.
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace swz {
namespace tcrate {

constexpr int kThreads = 128;
constexpr int kDynSmem = 120 * 1024;  // more than half an SM's shared memory
constexpr int A_BYTES = 128 * 128;    // 128 rows of 128 bytes
constexpr int B_MAX_BYTES = 256 * 128;
constexpr int kTmemCols = 256;

// K-major operand, 128-byte swizzle: 128-byte rows, 8-row atoms 1024 bytes
// apart (stride byte offset), leading byte offset unused (encoded 1), the
// fixed 0b001 at bits 46-48, swizzle mode 2 at bits 61-63.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

template <int KIND, int CG, int S>
__global__ void __launch_bounds__(kThreads, 1)
    tc_rate_kernel(const uint4* __restrict__ A, const uint4* __restrict__ B, int n,
                   uint32_t idesc, int n_mma, uint64_t timeout_ns,
                   unsigned long long* __restrict__ times, float* __restrict__ D) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t run_ok;
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms are 1024-byte aligned
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t a_s = base, b_s = base + A_BYTES, bar = base + A_BYTES + B_MAX_BYTES;
  const uint32_t bar_full = bar + 8, bar_empty = bar + 16;  // stage mode
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;

  // operands: 16-byte chunk j of row r lands at chunk j ^ (r % 8) of that
  // row; a pair's CTA `rank` holds B rows rank * n/2 .. + n/2 - 1
  const int b_rows = n / CG;
  const uint4* Bl = B + size_t(rank) * b_rows * 8;
  const int a_chunks = 128 * 8, total = a_chunks + b_rows * 8;
  for (int q = threadIdx.x; q < total; q += kThreads) {
    const bool is_a = q < a_chunks;
    const int qq = is_a ? q : q - a_chunks;
    const int r = qq >> 3, j = qq & 7;
    const uint4 v = is_a ? A[qq] : Bl[qq];
    uint8_t* dst = gbase + (is_a ? 0 : A_BYTES) + r * 128 + ((j ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = v;
  }
  ptx::fence_proxy_async_smem();  // generic stores -> visible to the tensor core
  if (warp == 0) {
    ptx::tmem_alloc<CG>(ptx::smem_u32(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish<CG>();
  }
  if (threadIdx.x == 32) {
    ptx::mbar_init(bar, 1);
    ptx::mbar_init(bar_full, 1);
    ptx::mbar_init(bar_empty, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive(bar_full);  // its phase 0 completes: every test of parity 0 succeeds
    run_ok = 0;
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (threadIdx.x == 0 && rank == 0) {
    const uint64_t ad = sdesc_kmajor_sw128(a_s), bd = sdesc_kmajor_sw128(b_s);
    bool ok = true;
    const unsigned long long c0 = clock64();
    const uint64_t t0 = ptx::global_timer_ns();
    if constexpr (S == 0) {
      for (int i = 0; i < n_mma; ++i) {
        const uint64_t s = uint64_t(2 * (i & 3));  // one k-slice = 32 bytes = 2 units of 16
        ptx::mma<CG, KIND>(tmem, ad + s, bd + s, idesc, i ? 1u : 0u);
      }
    } else {
      const int stages = n_mma / S;
#pragma unroll 8
      for (int st = 0; st < stages; ++st) {
        if (ok && !ptx::mbar_test_wait(bar_full, 0)) ok = false;  // never fails
        ptx::tc_fence_after();
#pragma unroll
        for (int i = 0; i < S; ++i) {
          const uint64_t s = uint64_t(2 * (i & 3));
          ptx::mma<CG, KIND>(tmem, ad + s, bd + s, idesc, (st | i) ? 1u : 0u);
        }
        if constexpr (CG == 2) ptx::mma_commit_pair(bar_empty, 0x1);
        else ptx::mma_commit(bar_empty);
      }
    }
    if constexpr (CG == 2) ptx::mma_commit_pair(bar, 0x1);
    else ptx::mma_commit(bar);
    const uint64_t t_issued = ptx::global_timer_ns();
    bool done = false;
    while (!(done = ptx::mbar_try_wait(bar, 0)) &&
           ptx::global_timer_ns() - t_issued < timeout_ns) {
    }
    const uint64_t t1 = ptx::global_timer_ns();
    const unsigned long long c1 = clock64();
    if (!done) {  // expired: give the tensor core one more bounded wait before freeing TMEM
      while (!ptx::mbar_try_wait(bar, 0) && ptx::global_timer_ns() - t1 < timeout_ns) {
      }
    }
    unsigned long long* o = times + 4ull * (blockIdx.x / CG);
    o[0] = c1 - c0;
    o[1] = t1 - t0;
    o[2] = sm_id();
    o[3] = (done && ok) ? 0ull : 1ull;
    run_ok = done ? 1u : 0u;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  if (D != nullptr && blockIdx.x == 0 && run_ok) {
    // warp w reads TMEM lanes (rows) 32w .. 32w + 31
    const uint32_t row = warp * 32u + lane;
    for (int c = 0; c < n; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(tmem + ((warp * 32u) << 16) + uint32_t(c), r);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) D[size_t(row) * n + c + j] = __uint_as_float(r[j]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the peer's accumulator rows and commits are the leader's: neither CTA of a
  // pair frees TMEM or leaves before both are done
  if constexpr (CG == 2) ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<CG>(tmem, kTmemCols);
  }
}

// tcgen05.mma instruction descriptor, A and B K-major, D fp32 (same fields as
// the GEMM's): bits 4-5 D format, 7-9 / 10-12 A / B format, 17-22 N >> 3,
// 24-28 M >> 4.
constexpr uint32_t idesc_kmajor(int dtype, int m, int n) {
  return (1u << 4) | (uint32_t(dtype) << 7) | (uint32_t(dtype) << 10) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

template <int KIND, int CG, int S>
int launch(const void* A, const void* B, int n, int dtype, int n_mma, int ctas,
           uint64_t timeout_ns, unsigned long long* times, float* D, cudaStream_t s) {
  static bool attr_set[64] = {};
  static std::mutex mu;
  auto kern = tc_rate_kernel<KIND, CG, S>;
  int dev = 0;
  SWZ_CUDA_TRY(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return SWZ_EINVAL;
    if (!attr_set[dev]) {
      SWZ_CUDA_TRY(
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem));
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if constexpr (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  SWZ_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(A),
                                  static_cast<const uint4*>(B), n,
                                  idesc_kmajor(dtype, 128 * CG, n), n_mma, timeout_ns, times, D));
  return SWZ_OK;
}

// the instance for (kind, pair, MMAs per stage)
template <int KIND, int CG>
int launch_stage(int S, const void* A, const void* B, int n, int dtype, int n_mma, int ctas,
                 uint64_t timeout_ns, unsigned long long* times, float* D, cudaStream_t s) {
  switch (S) {
    case 0: return launch<KIND, CG, 0>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, D, s);
    case 4: return launch<KIND, CG, 4>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, D, s);
    case 8: return launch<KIND, CG, 8>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, D, s);
    case 16: return launch<KIND, CG, 16>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, D, s);
    default: return SWZ_EINVAL;
  }
}

}  // namespace tcrate
}  // namespace swz

extern "C" int swz_tc_rate_ex(int dtype, int n, int cta_pair, int mmas_per_stage, const void* A,
                              const void* B, int n_mma, int num_ctas, uint64_t* d_times,
                              float* d_D, void* stream) {
  using namespace swz;
  if (dtype != SWZ_F16 && dtype != SWZ_BF16 && dtype != SWZ_TF32) return SWZ_EINVAL;
  if (cta_pair != 0 && cta_pair != 1) return SWZ_EINVAL;
  const int S = mmas_per_stage;
  if (S != 0 && S != 4 && S != 8 && S != 16) return SWZ_EINVAL;
  if (cta_pair ? (n != 128 && n != 256) : (n != 64 && n != 128 && n != 256)) return SWZ_EINVAL;
  if (n_mma < 1 || n_mma > (1 << 24) || num_ctas < 0) return SWZ_EINVAL;
  if (S != 0 && n_mma % S != 0) return SWZ_EINVAL;
  if (!A || !B || !d_times || !aligned16(A) || !aligned16(B) ||
      (reinterpret_cast<uintptr_t>(d_times) & 7u) != 0)
    return SWZ_EINVAL;
  if (d_D && !aligned4(d_D)) return SWZ_EINVAL;
  // TF32 is measured back to back on one CTA only
  if (dtype == SWZ_TF32 && (cta_pair || S != 0)) return SWZ_EUNSUPPORTED;
  DeviceInfo dev{};
  int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  const int cg = cta_pair ? 2 : 1;
  const int ctas = num_ctas ? num_ctas : dev.num_sms / cg * cg;
  if (ctas > dev.num_sms || ctas % cg != 0) return SWZ_EINVAL;  // one CTA per SM, whole pairs
  // the issue loop is bounded by the tensor core itself; the wait after it
  // covers only the last instructions in flight
  const uint64_t timeout_ns = 2000000000ull;
  auto* times = reinterpret_cast<unsigned long long*>(d_times);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SWZ_TF32)
    return tcrate::launch<1, 1, 0>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, d_D, s);
  if (cta_pair)
    return tcrate::launch_stage<0, 2>(S, A, B, n, dtype, n_mma, ctas, timeout_ns, times, d_D, s);
  return tcrate::launch_stage<0, 1>(S, A, B, n, dtype, n_mma, ctas, timeout_ns, times, d_D, s);
}

extern "C" int swz_tc_rate(int dtype, int n, const void* A, const void* B, int n_mma,
                           int num_ctas, uint64_t* d_times, float* d_D, void* stream) {
  return swz_tc_rate_ex(dtype, n, 0, 0, A, B, n_mma, num_ctas, d_times, d_D, stream);
}
