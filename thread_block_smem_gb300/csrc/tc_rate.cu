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
// (n x 128 bytes, K-major) into the 128-byte-swizzled layout the GEMM uses;
// warp 0 allocates 256 TMEM columns; thread 0 issues n_mma MMAs of shape
// 128 x n x k (k = 16 for fp16/bf16, 8 for TF32) cycling through the four
// k-slices of the 128-byte rows, all into one fp32 accumulator, commits,
// waits (bounded) and records its cycle and time spans.  CTA 0 then copies
// the accumulator out so a caller can check the MMAs really ran: with n_mma
// a multiple of 4 it holds (n_mma / 4) * A * B^T.
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

template <int KIND>
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
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;

  // operands: 16-byte chunk j of row r lands at chunk j ^ (r % 8) of that row
  const int a_chunks = 128 * 8, total = a_chunks + n * 8;
  for (int q = threadIdx.x; q < total; q += kThreads) {
    const bool is_a = q < a_chunks;
    const int qq = is_a ? q : q - a_chunks;
    const int r = qq >> 3, j = qq & 7;
    const uint4 v = is_a ? A[qq] : B[qq];
    uint8_t* dst = gbase + (is_a ? 0 : A_BYTES) + r * 128 + ((j ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = v;
  }
  ptx::fence_proxy_async_smem();  // generic stores -> visible to the tensor core
  if (warp == 0) {
    ptx::tmem_alloc<1>(ptx::smem_u32(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish<1>();
  }
  if (threadIdx.x == 32) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
    run_ok = 0;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (threadIdx.x == 0) {
    const uint64_t ad = sdesc_kmajor_sw128(a_s), bd = sdesc_kmajor_sw128(b_s);
    const unsigned long long c0 = clock64();
    const uint64_t t0 = ptx::global_timer_ns();
    for (int i = 0; i < n_mma; ++i) {
      const uint64_t s = uint64_t(2 * (i & 3));  // one k-slice = 32 bytes = 2 units of 16
      ptx::mma<1, KIND>(tmem, ad + s, bd + s, idesc, i ? 1u : 0u);
    }
    ptx::mma_commit(bar);
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
    unsigned long long* o = times + 4ull * blockIdx.x;
    o[0] = c1 - c0;
    o[1] = t1 - t0;
    o[2] = sm_id();
    o[3] = done ? 0ull : 1ull;
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
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<1>(tmem, kTmemCols);
  }
}

// tcgen05.mma instruction descriptor, A and B K-major, D fp32 (same fields as
// the GEMM's): bits 4-5 D format, 7-9 / 10-12 A / B format, 17-22 N >> 3,
// 24-28 M >> 4.
constexpr uint32_t idesc_kmajor(int dtype, int m, int n) {
  return (1u << 4) | (uint32_t(dtype) << 7) | (uint32_t(dtype) << 10) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

template <int KIND>
int launch(const void* A, const void* B, int n, int dtype, int n_mma, int ctas,
           uint64_t timeout_ns, unsigned long long* times, float* D, cudaStream_t s) {
  static bool attr_set[64] = {};
  static std::mutex mu;
  int dev = 0;
  SWZ_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return SWZ_EINVAL;
  if (!attr_set[dev]) {
    SWZ_CUDA_TRY(cudaFuncSetAttribute(tc_rate_kernel<KIND>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem));
    attr_set[dev] = true;
  }
  tc_rate_kernel<KIND><<<ctas, kThreads, kDynSmem, s>>>(
      static_cast<const uint4*>(A), static_cast<const uint4*>(B), n, idesc_kmajor(dtype, 128, n),
      n_mma, timeout_ns, times, D);
  SWZ_CUDA_TRY(cudaGetLastError());
  return SWZ_OK;
}

}  // namespace tcrate
}  // namespace swz

extern "C" int swz_tc_rate(int dtype, int n, const void* A, const void* B, int n_mma,
                           int num_ctas, uint64_t* d_times, float* d_D, void* stream) {
  using namespace swz;
  if (dtype != SWZ_F16 && dtype != SWZ_BF16 && dtype != SWZ_TF32) return SWZ_EINVAL;
  if (n != 64 && n != 128 && n != 256) return SWZ_EINVAL;
  if (n_mma < 1 || n_mma > (1 << 24) || num_ctas < 0) return SWZ_EINVAL;
  if (!A || !B || !d_times || !aligned16(A) || !aligned16(B) ||
      (reinterpret_cast<uintptr_t>(d_times) & 7u) != 0)
    return SWZ_EINVAL;
  if (d_D && !aligned4(d_D)) return SWZ_EINVAL;
  DeviceInfo dev{};
  int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  const int ctas = num_ctas ? num_ctas : dev.num_sms;
  if (ctas > dev.num_sms) return SWZ_EINVAL;  // at most one CTA per SM
  // the issue loop is bounded by the tensor core itself; the wait after it
  // covers only the last instructions in flight
  const uint64_t timeout_ns = 2000000000ull;
  auto* times = reinterpret_cast<unsigned long long*>(d_times);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SWZ_TF32)
    return tcrate::launch<1>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, d_D, s);
  return tcrate::launch<0>(A, B, n, dtype, n_mma, ctas, timeout_ns, times, d_D, s);
}
