// noalloc.cu -- swz_gemm_streamk_noalloc: the Stream-K GEMM with its scratch
// in a device array built into the library, for callers that cannot
// allocate device memory (plugin hosts that hand over only input and output
// buffers, services on a fixed memory budget whose allocator belongs to
// someone else, loops that must not call cudaMalloc because it synchronises
// the device).  The source pages have no counterpart of this entry point.
//
// The array lives in this translation unit only, so the 40 MiB are held by a
// GPU once this file's code is loaded there (at the latest on the first call
// of the entry point) and stay held until the process exits.  That covers
// the largest launch with the default program count on a GB300: two
// workspace slots per program of 128 x 256 FP32 partial sums (1-CTA tiles,
// 152 programs, or 76 CTA pairs), 38 MiB, and their flags.
#include <mutex>

#include "common.h"

namespace {

// Scratch of swz_gemm_streamk_noalloc.  In host code this name is only a
// stand-in for the device array (passing it to a kernel would be wrong); the
// device address comes from cudaGetSymbolAddress in scratch_address().
static __device__ __align__(256) unsigned char noalloc_scratch[SWZ_NOALLOC_SCRATCH_BYTES];

// Device address of noalloc_scratch on `device`, which must be current.
// Looked up once per device and kept for the life of the process: it does
// not survive cudaDeviceReset (the array is allocated anew in the next
// context), so the entry point must not be called after a reset.
int scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  if (device < 0 || device >= 64) return SWZ_EINVAL;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch);
    if (e != cudaSuccess) return swz::cuda_fail(e);
    if (!p) return swz::cuda_fail(cudaErrorInvalidSymbol);
    addr[device] = p;
  }
  *out = addr[device];
  return SWZ_OK;
}

}  // namespace

extern "C" int swz_gemm_streamk_noalloc(const void* A, const void* B, float* C, int M, int N,
                                        int K, int order, int group, const swz_gemm_opts* opts,
                                        void* stream) {
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  o.stream_k = 1;
  o.d_workspace = nullptr;
  o.workspace_bytes = 0;
  if (M < 0 || N < 0 || K < 0) return SWZ_EINVAL;
  if (M > 0 && N > 0 && K > 0) {
    uint64_t flag_bytes = 0, total = 0;
    int rc = swz::gemm_sk_workspace_split(M, N, K, 1, o, &flag_bytes, &total);
    if (rc != SWZ_OK) return rc;
    if (total > SWZ_NOALLOC_SCRATCH_BYTES) return SWZ_ESCRATCH;
    if (total > 0) {
      swz::DeviceInfo dev{};
      rc = swz::current_device(&dev);
      if (rc != SWZ_OK) return rc;
      void* scratch = nullptr;
      rc = scratch_address(dev.device, &scratch);
      if (rc != SWZ_OK) return rc;
      o.d_workspace = scratch;
      o.workspace_bytes = SWZ_NOALLOC_SCRATCH_BYTES;
    }
  }
  // The flags must not hold a value this launch could mistake for a
  // finished piece: the launch clears them on the stream first (the partial
  // sums need no clearing), once every argument check has passed.
  return swz::gemm_ex(A, B, C, M, N, K, order, group, 1, &o, stream, true);
}
