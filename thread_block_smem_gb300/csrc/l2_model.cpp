// l2_model.cpp -- host-side offline L2 hit-rate model of a tile order.
//
// The model of Lei Mao, "CUDA Thread Block Swizzle", benchmark section: the
// L2 holds whole operand tiles under a byte budget with least-recently-used
// replacement (a hit refreshes the tile; a miss inserts it, then the oldest
// tiles are dropped while the budget is exceeded and more than one tile is
// held).  Program ids are taken in waves of `concurrency`; inside a wave, for
// every K step, each tile of the wave touches its A tile (m, k) and then its
// B tile (k, n).  With CTA clusters of `cluster_m` CTAs along M, the order
// runs on cluster tiles and each cluster tile contributes its CTA tiles in
// rank order (TVM TIRx "ClusterPersistentScheduler2D", Example 2).
//
// l2_partitions > 1 is not the page's model but a reading of a GPU whose L2
// is split into that many halves (one per die, as on GB300): the SMs of
// every die read every operand line of a wave, and each die's half keeps its
// own copy of what its SMs read, so each half replays the whole trace with
// 1 / l2_partitions of the capacity.  The prediction is that of one half.
//
// k_alternate = 1 is the K order of the library's persistent GEMM, not the
// page's: the tiles of odd waves take the K steps from the last to the first.
#include <stdint.h>

#include <list>
#include <unordered_map>
#include <utility>
#include <vector>

#include "swz.h"
#include "tile_order.cuh"

namespace {

class LruBytes {
 public:
  explicit LruBytes(int64_t cap) : cap_(cap) {}

  void touch(uint64_t key, int64_t bytes) {
    auto it = where_.find(key);
    if (it != where_.end()) {
      ++hits_;
      order_.splice(order_.end(), order_, it->second);
      return;
    }
    ++misses_;
    miss_bytes_ += bytes;
    order_.emplace_back(key, bytes);
    where_.emplace(key, std::prev(order_.end()));
    held_ += bytes;
    while (held_ > cap_ && order_.size() > 1) {
      held_ -= order_.front().second;
      where_.erase(order_.front().first);
      order_.pop_front();
    }
  }

  int64_t hits() const { return hits_; }
  int64_t misses() const { return misses_; }
  int64_t miss_bytes() const { return miss_bytes_; }

 private:
  int64_t cap_, held_ = 0, hits_ = 0, misses_ = 0, miss_bytes_ = 0;
  std::list<std::pair<uint64_t, int64_t>> order_;
  std::unordered_map<uint64_t, std::list<std::pair<uint64_t, int64_t>>::iterator> where_;
};

inline uint64_t key_a(uint64_t m, uint64_t k) { return (m << 32) | k; }
inline uint64_t key_b(uint64_t k, uint64_t n) { return (uint64_t(1) << 63) | (n << 32) | k; }

}  // namespace

extern "C" int swz_l2_model_bytes(int order, int group, int M, int N, int K, int tile_m,
                                  int tile_n, int tile_k, int elem_bytes, int64_t l2_bytes,
                                  int l2_partitions, int k_alternate, int concurrency,
                                  int cluster_m, int64_t* hits, int64_t* misses,
                                  int64_t* miss_bytes) {
  if (!swz::order_is_valid(order) || (swz::order_uses_group(order) && group < 1)) return SWZ_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || tile_m <= 0 || tile_n <= 0 || tile_k <= 0) return SWZ_EINVAL;
  if (elem_bytes <= 0 || l2_bytes < 0 || concurrency <= 0 || cluster_m <= 0) return SWZ_EINVAL;
  if (l2_partitions < 1 || (k_alternate != 0 && k_alternate != 1)) return SWZ_EINVAL;
  if (!hits || !misses || !miss_bytes) return SWZ_EINVAL;
  const int64_t span_m = int64_t(tile_m) * cluster_m;
  const uint32_t sm = uint32_t((int64_t(M) + span_m - 1) / span_m);
  const uint32_t gn = uint32_t((int64_t(N) + tile_n - 1) / tile_n);
  const uint32_t gk = uint32_t((int64_t(K) + tile_k - 1) / tile_k);
  const uint64_t units = uint64_t(sm) * gn;
  if (units * uint64_t(cluster_m) > (uint64_t(1) << 31)) return SWZ_EINVAL;
  const uint32_t g = swz::order_uses_group(order) ? uint32_t(group) : 1u;

  // CTA-tile sequence in program order
  std::vector<std::pair<uint32_t, uint32_t>> seq;
  seq.reserve(units * cluster_m);
  for (uint64_t w = 0; w < units; ++w) {
    const swz::TileCoord t = swz::tile_of(order, uint32_t(w), sm, gn, g);
    for (int r = 0; r < cluster_m; ++r) seq.emplace_back(t.m * uint32_t(cluster_m) + r, t.n);
  }
  const int64_t a_bytes = int64_t(tile_m) * tile_k * elem_bytes;
  const int64_t b_bytes = int64_t(tile_k) * tile_n * elem_bytes;
  LruBytes cache(l2_bytes / l2_partitions);
  for (size_t w0 = 0; w0 < seq.size(); w0 += size_t(concurrency)) {
    const size_t w1 = w0 + size_t(concurrency) < seq.size() ? w0 + size_t(concurrency) : seq.size();
    const bool descending = k_alternate && (w0 / size_t(concurrency)) % 2 == 1;
    for (uint32_t kk = 0; kk < gk; ++kk) {
      const uint32_t k = descending ? gk - 1 - kk : kk;
      for (size_t i = w0; i < w1; ++i) {
        cache.touch(key_a(seq[i].first, k), a_bytes);
        cache.touch(key_b(k, seq[i].second), b_bytes);
      }
    }
  }
  *hits = cache.hits();
  *misses = cache.misses();
  *miss_bytes = cache.miss_bytes();
  return SWZ_OK;
}

extern "C" int swz_l2_model(int order, int group, int M, int N, int K, int tile_m, int tile_n,
                            int tile_k, int elem_bytes, int64_t l2_bytes, int concurrency,
                            int cluster_m, int64_t* hits, int64_t* misses) {
  if (!hits || !misses) return SWZ_EINVAL;
  int64_t bytes = 0;
  return swz_l2_model_bytes(order, group, M, N, K, tile_m, tile_n, tile_k, elem_bytes, l2_bytes,
                            1, 0, concurrency, cluster_m, hits, misses, &bytes);
}
