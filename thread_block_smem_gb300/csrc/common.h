// common.h -- host-side helpers shared by the entry points of libswz.so:
// status codes, CUDA error capture and the device-architecture check.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "swz.h"

namespace swz {

// cudaError_t of the last failing CUDA call made by this thread.
int& last_cuda_error_slot();

// Records a failing CUDA call and maps it to SWZ_ECUDA.
inline int cuda_fail(cudaError_t e) {
  last_cuda_error_slot() = static_cast<int>(e);
  return SWZ_ECUDA;
}

#define SWZ_CUDA_TRY(expr)                       \
  do {                                           \
    cudaError_t swz_e_ = (expr);                 \
    if (swz_e_ != cudaSuccess) return ::swz::cuda_fail(swz_e_); \
  } while (0)

// Current device, its SM count and whether it is sm_103 (GB300).
struct DeviceInfo {
  int device;
  int num_sms;
  int l2_bytes;
  int cc_major, cc_minor;
};

// Fills `info` for the current device; SWZ_OK, SWZ_ECUDA or SWZ_EARCH.
int current_device(DeviceInfo* info, bool require_sm103 = true);

// True when `order` visits each tile of the gm x gn grid exactly once
// (host-side exhaustive check over all ids).
bool order_is_bijective(int order, uint32_t gm, uint32_t gn, uint32_t group);

// Stream-K workspace split of a launch: bytes of the flag block at the front
// and total bytes (both 0 when the launch needs no workspace).
int gemm_sk_workspace_split(int M, int N, int K, int persistent, const swz_gemm_opts& o,
                            uint64_t* flag_bytes, uint64_t* total_bytes);

// swz_gemm_ex; with clear_sk_flags a Stream-K launch clears its piece flags
// on the stream before it starts (always, not only under stream capture),
// after every argument check has passed.
int gemm_ex(const void* A, const void* B, float* C, int M, int N, int K, int order, int group,
            int persistent, const swz_gemm_opts* opts, void* stream, bool clear_sk_flags);

// The die of every SM of the current device (indexed by SM id; 0 or 1,
// all 0 on a single die), found by timing L2 hits: SWZ_OK, SWZ_ECUDA, or
// SWZ_EUNSUPPORTED when not every SM could be measured.
int die_of_sms(int num_sms, std::vector<uint8_t>* die_of_sm);

// The SM id of every CTA of one launch of `grid` CTAs in clusters of
// `cluster` with `threads` threads and `smem` bytes of dynamic shared memory.
int placement(int cluster, int threads, int smem, int grid, std::vector<uint32_t>* sm_of_cta);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace swz
