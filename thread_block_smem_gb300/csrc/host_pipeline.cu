// host_pipeline.cu -- swz_gemm_host: C = A * B from host buffers, with the
// host->device copies, the GEMM and the device->host copy overlapped.
//
// B is copied in whole first (every output row needs all of it).  A and C
// are cut into row slabs: while slab i is multiplied on the caller's stream,
// slab i+1 of A is copied in on an input stream and slab i-1 of C is copied
// out on an output stream.  Events order the three streams; the caller's
// stream waits for the last copy, so the call behaves like one operation on
// `stream`.  Each slab is an ordinary swz_gemm_ex launch on the slab's rows
// (the tile order applies within a slab).
#include <mutex>

#include "common.h"

namespace {

constexpr int kMaxSlabs = 64;

// Streams and events of the pipeline, created once per device and kept for
// the life of the process (no device memory).
struct PipelineRes {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, b_in = nullptr, done = nullptr;
  cudaEvent_t a_in[kMaxSlabs] = {}, c_ready[kMaxSlabs] = {};
};

std::mutex g_pipe_mu;  // serialises enqueueing on the shared streams/events

int resources(int device, PipelineRes** out) {
  static PipelineRes res[64];
  static bool ready[64] = {};
  if (device < 0 || device >= 64) return SWZ_EINVAL;
  PipelineRes& r = res[device];
  if (!ready[device]) {
    const unsigned ef = cudaEventDisableTiming;
    SWZ_CUDA_TRY(cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking));
    SWZ_CUDA_TRY(cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking));
    SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.start, ef));
    SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.b_in, ef));
    SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.done, ef));
    for (int i = 0; i < kMaxSlabs; ++i) {
      SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.a_in[i], ef));
      SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.c_ready[i], ef));
    }
    ready[device] = true;
  }
  *out = &r;
  return SWZ_OK;
}

}  // namespace

extern "C" int swz_gemm_host(const void* h_A, const void* h_B, float* h_C, int M, int N, int K,
                             int order, int group, const swz_gemm_opts* opts, void* d_A,
                             void* d_B, float* d_C, int slabs, void* stream) {
  if (M < 0 || N < 0 || K < 0 || slabs < 0 || slabs > kMaxSlabs) return SWZ_EINVAL;
  if (M == 0 || N == 0) return SWZ_OK;
  if (!h_C || !d_C || !swz::aligned16(d_C)) return SWZ_EINVAL;
  if (K > 0 && (!h_A || !h_B || !d_A || !d_B || !swz::aligned16(d_A) || !swz::aligned16(d_B)))
    return SWZ_EINVAL;
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  if (o.dtype != SWZ_F16 && o.dtype != SWZ_BF16 && o.dtype != SWZ_TF32) return SWZ_EINVAL;
  if (o.b_layout != SWZ_B_KN && o.b_layout != SWZ_B_NK) return SWZ_EINVAL;
  if (o.dtype == SWZ_TF32 && o.b_layout != SWZ_B_NK) return SWZ_EUNSUPPORTED;
  const size_t esize = o.dtype == SWZ_TF32 ? 4 : 2;  // fp32 (TF32) or fp16 / bf16
  const int per16 = int(16 / esize);
  if (N % 4 || (K > 0 && K % per16) || (o.b_layout == SWZ_B_KN && N % per16)) return SWZ_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // slab rows: a multiple of 256 (one cluster tile of rows) when possible
  const int S = slabs ? slabs : 4;
  int64_t rows = (int64_t(M) + S - 1) / S;
  rows = (rows + 255) / 256 * 256;
  const int nslab = int((int64_t(M) + rows - 1) / rows);

  // everything that can fail on the host is checked before enqueueing
  if (K > 0) {
    for (int i = 0; i < nslab; ++i) {
      const int mi = int(rows < int64_t(M) - i * rows ? rows : int64_t(M) - i * rows);
      int t_m = 0, t_n = 0, s_m = 0, s_n = 0, progs = 0;
      int rc = swz_gemm_plan(mi, N, K, 1, &o, &t_m, &t_n, &s_m, &s_n, &progs);
      if (rc != SWZ_OK) return rc;
      if (order == SWZ_MORTON || order == SWZ_XOR) {
        rc = swz_is_bijective(order, s_m, s_n, group);
        if (rc < 0) return rc;
        if (rc == 0) return SWZ_ENOTBIJECTIVE;
      }
    }
  }
  swz::DeviceInfo dev{};
  int rc = swz::current_device(&dev);
  if (rc != SWZ_OK) return rc;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  PipelineRes* r = nullptr;
  rc = resources(dev.device, &r);
  if (rc != SWZ_OK) return rc;

  if (K == 0) {  // C = 0: clear on the device, copy out
    SWZ_CUDA_TRY(cudaMemsetAsync(d_C, 0, size_t(M) * N * sizeof(float), s));
    SWZ_CUDA_TRY(cudaMemcpyAsync(h_C, d_C, size_t(M) * N * sizeof(float),
                                 cudaMemcpyDeviceToHost, s));
    return SWZ_OK;
  }

  SWZ_CUDA_TRY(cudaEventRecord(r->start, s));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(r->in, r->start, 0));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(r->out, r->start, 0));
  SWZ_CUDA_TRY(cudaMemcpyAsync(d_B, h_B, size_t(K) * N * esize, cudaMemcpyHostToDevice, r->in));
  SWZ_CUDA_TRY(cudaEventRecord(r->b_in, r->in));
  for (int i = 0; i < nslab; ++i) {
    const int64_t r0 = i * rows;
    const int64_t mi = rows < M - r0 ? rows : M - r0;
    const size_t a_off = size_t(r0) * K * esize;
    SWZ_CUDA_TRY(cudaMemcpyAsync(static_cast<char*>(d_A) + a_off,
                                 static_cast<const char*>(h_A) + a_off, size_t(mi) * K * esize,
                                 cudaMemcpyHostToDevice, r->in));
    SWZ_CUDA_TRY(cudaEventRecord(r->a_in[i], r->in));
  }
  SWZ_CUDA_TRY(cudaStreamWaitEvent(s, r->b_in, 0));
  for (int i = 0; i < nslab; ++i) {
    const int64_t r0 = i * rows;
    const int mi = int(rows < M - r0 ? rows : M - r0);
    SWZ_CUDA_TRY(cudaStreamWaitEvent(s, r->a_in[i], 0));
    rc = swz_gemm_ex(static_cast<const char*>(d_A) + size_t(r0) * K * esize, d_B,
                     d_C + size_t(r0) * N, mi, N, K, order, group, 1, &o, stream);
    if (rc != SWZ_OK) return rc;
    SWZ_CUDA_TRY(cudaEventRecord(r->c_ready[i], s));
    SWZ_CUDA_TRY(cudaStreamWaitEvent(r->out, r->c_ready[i], 0));
    SWZ_CUDA_TRY(cudaMemcpyAsync(h_C + size_t(r0) * N, d_C + size_t(r0) * N,
                                 size_t(mi) * N * sizeof(float), cudaMemcpyDeviceToHost, r->out));
  }
  SWZ_CUDA_TRY(cudaEventRecord(r->done, r->out));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(s, r->done, 0));
  return SWZ_OK;
}
