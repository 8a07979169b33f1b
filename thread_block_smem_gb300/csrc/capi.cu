// capi.cu -- status strings, device queries, the host bijectivity check and
// the tile-map kernel of libswz.so.
//
// swz_tile_map evaluates, on the device, the tile-order function the GEMM's
// scheduler uses (Lei Mao, "CUDA Thread Block Swizzle", tile-order sections;
// TVM TIRx "ClusterPersistentScheduler2D", "Serpentine Mode"), so that the
// map can be compared bit for bit with an independent implementation.
#include <mutex>
#include <vector>

#include "common.h"
#include "tile_order.cuh"

namespace swz {

int& last_cuda_error_slot() {
  static thread_local int slot = 0;
  return slot;
}

int current_device(DeviceInfo* info, bool require_sm103) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  SWZ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (have[dev]) {
      *info = cache[dev];
    } else {
      DeviceInfo d{};
      d.device = dev;
      SWZ_CUDA_TRY(cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev));
      SWZ_CUDA_TRY(cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev));
      SWZ_CUDA_TRY(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
      SWZ_CUDA_TRY(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
      cache[dev] = d;
      have[dev] = true;
      *info = d;
    }
  } else {
    return SWZ_EINVAL;
  }
  if (require_sm103 && !(info->cc_major == 10 && info->cc_minor == 3)) return SWZ_EARCH;
  return SWZ_OK;
}

// Marks every tile the order reaches; true when all gm*gn are reached once.
bool order_is_bijective(int order, uint32_t gm, uint32_t gn, uint32_t group) {
  const uint64_t tiles = uint64_t(gm) * gn;
  std::vector<uint8_t> seen(tiles, 0);
  for (uint64_t id = 0; id < tiles; ++id) {
    const TileCoord t = tile_of(order, uint32_t(id), gm, gn, group);
    if (t.m >= gm || t.n >= gn) return false;
    uint8_t& s = seen[uint64_t(t.m) * gn + t.n];
    if (s) return false;
    s = 1;
  }
  return true;
}

__global__ void tile_map_kernel(int order, uint32_t gm, uint32_t gn, uint32_t group,
                                uint32_t tiles, int32_t* __restrict__ out_m,
                                int32_t* __restrict__ out_n) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t id = blockIdx.x * blockDim.x + threadIdx.x; id < tiles; id += stride) {
    const TileCoord t = tile_of(order, id, gm, gn, group);
    out_m[id] = int32_t(t.m);
    out_n[id] = int32_t(t.n);
  }
}

}  // namespace swz

using namespace swz;

extern "C" const char* swz_strerror(int status) {
  switch (status) {
    case SWZ_OK: return "success";
    case SWZ_EINVAL: return "invalid argument (null pointer, size, enum or alignment)";
    case SWZ_ENOTBIJECTIVE: return "tile order is not a permutation of this tile grid";
    case SWZ_EARCH: return "current device is not sm_103 (GB300)";
    case SWZ_ECUDA: return "CUDA runtime call failed (see swz_last_cuda_error)";
    case SWZ_ETIMEOUT: return "a bounded device wait expired";
    case SWZ_EUNSUPPORTED: return "configuration not supported";
    case SWZ_ESCRATCH: return "launch needs more scratch than the built-in scratch area holds";
    default: return "unknown status";
  }
}

extern "C" int swz_last_cuda_error(void) { return last_cuda_error_slot(); }

extern "C" int swz_device_info(int* num_sms, int* l2_bytes, int* cc_major, int* cc_minor) {
  DeviceInfo d{};
  const int rc = current_device(&d, /*require_sm103=*/false);
  if (rc != SWZ_OK) return rc;
  if (num_sms) *num_sms = d.num_sms;
  if (l2_bytes) *l2_bytes = d.l2_bytes;
  if (cc_major) *cc_major = d.cc_major;
  if (cc_minor) *cc_minor = d.cc_minor;
  return SWZ_OK;
}

extern "C" int swz_is_bijective(int order, int grid_m, int grid_n, int group) {
  if (!order_is_valid(order) || grid_m <= 0 || grid_n <= 0) return SWZ_EINVAL;
  if (int64_t(grid_m) * grid_n > INT32_MAX) return SWZ_EINVAL;
  if (order_uses_group(order) && group < 1) return SWZ_EINVAL;
  return order_is_bijective(order, uint32_t(grid_m), uint32_t(grid_n), uint32_t(group)) ? 1 : 0;
}

extern "C" int swz_tile_map(int order, int grid_m, int grid_n, int group, int32_t* d_m,
                            int32_t* d_n, void* stream) {
  if (!order_is_valid(order) || grid_m <= 0 || grid_n <= 0 || !d_m || !d_n) return SWZ_EINVAL;
  if (int64_t(grid_m) * grid_n > INT32_MAX) return SWZ_EINVAL;
  if (order_uses_group(order) && group < 1) return SWZ_EINVAL;
  DeviceInfo dev{};
  const int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  const uint32_t tiles = uint32_t(grid_m) * uint32_t(grid_n);
  const int threads = 256;
  const uint32_t want = (tiles + threads - 1) / threads;
  const uint32_t cap = uint32_t(dev.num_sms) * 8u;
  const uint32_t blocks = want < cap ? want : cap;
  tile_map_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      order, uint32_t(grid_m), uint32_t(grid_n), uint32_t(order_uses_group(order) ? group : 1),
      tiles, d_m, d_n);
  SWZ_CUDA_TRY(cudaGetLastError());
  return SWZ_OK;
}
