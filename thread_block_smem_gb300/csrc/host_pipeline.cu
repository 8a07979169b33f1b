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
  cudaEvent_t panel_in[kMaxSlabs] = {};  // B column panels (tiled pipeline)
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
      SWZ_CUDA_TRY(cudaEventCreateWithFlags(&r.panel_in[i], ef));
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

// swz_gemm_host_tiled -- the same product, with C cut into g x g blocks that
// are finished in a growing square: after row slab t of A and column panel t
// of B have arrived, blocks (t, 0..t) and (0..t-1, t) are computed and copied
// out.  C thus starts leaving while A and B are still arriving, which the
// row-slab pipeline above cannot do (every C row needs all of B).  Column
// panels of a K x N B are gathered into packed K x N_j staging panels by
// pitched copies (a N x K B needs none: its panels are contiguous rows); C
// blocks are computed into packed staging blocks and scattered into h_C by
// pitched copies.
extern "C" int swz_gemm_host_tiled(const void* h_A, const void* h_B, float* h_C, int M, int N,
                                   int K, int order, int group, const swz_gemm_opts* opts,
                                   void* d_A, void* d_B, float* d_C, int blocks,
                                   void* stream) {
  if (M < 0 || N < 0 || K < 0 || blocks < 0 || blocks > 8) return SWZ_EINVAL;
  if (M == 0 || N == 0) return SWZ_OK;
  if (!h_C || !d_C || !swz::aligned16(d_C)) return SWZ_EINVAL;
  if (K > 0 && (!h_A || !h_B || !d_A || !d_B || !swz::aligned16(d_A) || !swz::aligned16(d_B)))
    return SWZ_EINVAL;
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  if (o.dtype != SWZ_F16 && o.dtype != SWZ_BF16 && o.dtype != SWZ_TF32) return SWZ_EINVAL;
  if (o.b_layout != SWZ_B_KN && o.b_layout != SWZ_B_NK) return SWZ_EINVAL;
  if (o.dtype == SWZ_TF32 && o.b_layout != SWZ_B_NK) return SWZ_EUNSUPPORTED;
  const size_t esize = o.dtype == SWZ_TF32 ? 4 : 2;
  const int per16 = int(16 / esize);
  if (N % 4 || (K > 0 && K % per16) || (o.b_layout == SWZ_B_KN && N % per16)) return SWZ_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // block boundaries, multiples of 256 (one cluster tile); trailing blocks
  // may be empty when M or N is small
  const int g = blocks ? blocks : 4;
  const int64_t rw = ((int64_t(M) + g - 1) / g + 255) / 256 * 256;
  const int64_t cw = ((int64_t(N) + g - 1) / g + 255) / 256 * 256;
  int64_t r[9], c[9];
  for (int t = 0; t <= g; ++t) {
    r[t] = t * rw < M ? t * rw : M;
    c[t] = t * cw < N ? t * cw : N;
  }
  // blocks in the order they are computed: the growing square
  int bi[64], bj[64], nb = 0;
  for (int t = 0; t < g; ++t) {
    for (int j = 0; j <= t; ++j) { bi[nb] = t; bj[nb] = j; ++nb; }
    for (int i = 0; i < t; ++i) { bi[nb] = i; bj[nb] = t; ++nb; }
  }

  // everything that can fail on the host is checked before enqueueing
  if (K > 0) {
    for (int b = 0; b < nb; ++b) {
      const int mi = int(r[bi[b] + 1] - r[bi[b]]), nj = int(c[bj[b] + 1] - c[bj[b]]);
      if (mi == 0 || nj == 0) continue;
      int t_m = 0, t_n = 0, s_m = 0, s_n = 0, progs = 0;
      int rc = swz_gemm_plan(mi, nj, K, 1, &o, &t_m, &t_n, &s_m, &s_n, &progs);
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
  PipelineRes* res = nullptr;
  rc = resources(dev.device, &res);
  if (rc != SWZ_OK) return rc;

  if (K == 0) {  // C = 0: clear on the device, copy out
    SWZ_CUDA_TRY(cudaMemsetAsync(d_C, 0, size_t(M) * N * sizeof(float), s));
    SWZ_CUDA_TRY(cudaMemcpyAsync(h_C, d_C, size_t(M) * N * sizeof(float),
                                 cudaMemcpyDeviceToHost, s));
    return SWZ_OK;
  }

  const char* hA = static_cast<const char*>(h_A);
  const char* hB = static_cast<const char*>(h_B);
  char* dA = static_cast<char*>(d_A);
  char* dB = static_cast<char*>(d_B);
  SWZ_CUDA_TRY(cudaEventRecord(res->start, s));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(res->in, res->start, 0));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(res->out, res->start, 0));
  // inputs: A slab t, then B panel t, for t = 0, 1, ...
  for (int t = 0; t < g; ++t) {
    const int64_t mi = r[t + 1] - r[t], nj = c[t + 1] - c[t];
    if (mi > 0) {
      const size_t off = size_t(r[t]) * K * esize;
      SWZ_CUDA_TRY(cudaMemcpyAsync(dA + off, hA + off, size_t(mi) * K * esize,
                                   cudaMemcpyHostToDevice, res->in));
    }
    SWZ_CUDA_TRY(cudaEventRecord(res->a_in[t], res->in));
    if (nj > 0) {
      char* dst = dB + size_t(c[t]) * K * esize;  // packed panel: K x nj (or nj x K)
      if (o.b_layout == SWZ_B_NK)
        SWZ_CUDA_TRY(cudaMemcpyAsync(dst, hB + size_t(c[t]) * K * esize, size_t(nj) * K * esize,
                                     cudaMemcpyHostToDevice, res->in));
      else
        SWZ_CUDA_TRY(cudaMemcpy2DAsync(dst, size_t(nj) * esize, hB + size_t(c[t]) * esize,
                                       size_t(N) * esize, size_t(nj) * esize, size_t(K),
                                       cudaMemcpyHostToDevice, res->in));
    }
    SWZ_CUDA_TRY(cudaEventRecord(res->panel_in[t], res->in));
  }
  // blocks: GEMM on the caller's stream, copy-out on the output stream
  for (int b = 0; b < nb; ++b) {
    const int i = bi[b], j = bj[b];
    const int mi = int(r[i + 1] - r[i]), nj = int(c[j + 1] - c[j]);
    if (mi == 0 || nj == 0) continue;
    SWZ_CUDA_TRY(cudaStreamWaitEvent(s, res->a_in[i], 0));
    SWZ_CUDA_TRY(cudaStreamWaitEvent(s, res->panel_in[j], 0));
    float* blk = d_C + size_t(r[i]) * N + size_t(mi) * size_t(c[j]);  // packed mi x nj
    rc = swz_gemm_ex(dA + size_t(r[i]) * K * esize, dB + size_t(c[j]) * K * esize, blk, mi, nj,
                     K, order, group, 1, &o, stream);
    if (rc != SWZ_OK) return rc;
    SWZ_CUDA_TRY(cudaEventRecord(res->c_ready[b], s));
    SWZ_CUDA_TRY(cudaStreamWaitEvent(res->out, res->c_ready[b], 0));
    SWZ_CUDA_TRY(cudaMemcpy2DAsync(h_C + size_t(r[i]) * N + size_t(c[j]), size_t(N) * sizeof(float),
                                   blk, size_t(nj) * sizeof(float), size_t(nj) * sizeof(float),
                                   size_t(mi), cudaMemcpyDeviceToHost, res->out));
  }
  SWZ_CUDA_TRY(cudaEventRecord(res->done, res->out));
  SWZ_CUDA_TRY(cudaStreamWaitEvent(s, res->done, 0));
  return SWZ_OK;
}
