// gemm.cu -- C = A * B (fp16/bf16 in, fp32 accumulate and out) on sm_103a
// with a selectable thread-block swizzle and a persistent tile scheduler.
//
// What it computes: the masked tiled GEMM of Lei Mao, "CUDA Thread Block
// Swizzle" (benchmark section: program id -> output tile through the chosen
// tile order, a K loop per tile, masked loads and stores, persistent launch =
// each program takes tile ids pid, pid + P, pid + 2P, ...).  The scheduler is
// the work-index stride of TVM TIRx "ClusterPersistentScheduler2D"
// (work_idx = cluster_id + i * num_clusters, cluster tiles split into CTA
// tiles as in its "Example 2: 2SM GEMM").  Operands are staged with the
// 128-byte TMA swizzle of WHC, "CUDA Swizzle & bank conflict", section
// "Hopper TMA 的 swizzling" (16-byte chunk index XOR row mod 8 inside each
// 1024-byte atom), which the tensor cores read without bank conflicts.
//
// Design (GB300 / sm_103a):
//   * 192 threads per CTA, one CTA per SM.  Warp 0: TMA producer.  Warp 1:
//     TMEM allocator and (one lane) tcgen05.mma issuer.  Warps 2-5: epilogue
//     (warp w reads TMEM lanes 32*(w%4) .. +31).
//   * K is consumed in stages of KA 128-byte atoms per operand row (64 fp16
//     / bf16 or 32 TF32 elements per atom; KA = 1 for 256-wide tiles, 2 for
//     128-wide ones) through a ring of STAGES shared-memory stages guarded by
//     full/empty mbarriers.  A: 128 rows, K-major.  B: BN_LOCAL columns,
//     N-major (B given K x N, 64-column boxes) or K-major (B given N x K).
//     The swizzle span (128, 64 or 32 bytes) is a template parameter; the
//     64- and 32-byte spans split each 128-byte row into column groups.
//   * The accumulator lives in TMEM, double-buffered (2 x BN fp32 columns),
//     so the epilogue of tile i overlaps the MMAs of tile i+1.  When a tile
//     follows, the epilogue spreads its C stores (4 KB TMA boxes) over part
//     of the next tile instead of issuing them in one burst that would
//     share the TMA unit with that tile's first operand loads.
//   * CTA pair (PAIR): 2-CTA cluster, tcgen05 cta_group::2, MMA 256 x BN.
//     Each CTA loads its own 128 rows of A and its half of B's columns;
//     the leader issues the MMAs and its commits are multicast to both CTAs.
//   * Work items come from the static schedule (Schedule: work_idx striding,
//     optional Stream-K tail, optional split of the units between the two
//     dies) or, with DYN, from an atomic counter published one item ahead to
//     all roles through a shared-memory ring.  The pieces of a Stream-K tail
//     come first; their partial sums are published to a workspace and
//     reduced by the tiles' participants while the whole tiles run.
//   * Every wait is bounded (globaltimer); on expiry the kernel records
//     SWZ_ETIMEOUT in a device status word, drains what it issued, frees TMEM
//     and returns.
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace swz {

__device__ unsigned int g_status_word;  // nonzero: a bounded wait expired

namespace gemm {

constexpr int BM = 128;        // CTA tile rows = TMEM lanes
constexpr int BK = 64;         // K elements per stage, 16-bit operands (128-byte rows)
// With 32-bit (TF32) operands a stage holds 32 K elements: the same 128-byte
// rows, so every byte offset below is shared by both kinds.
template <int KIND>
constexpr int bk_elems() { return KIND == 0 ? 64 : 32; }
// 128-byte K atoms per stage with the 128-byte span, by tile width: a stage
// of KA atoms carries 4 * KA MMAs per barrier round trip of the issuing
// thread, whose per-stage overhead (~300 cycles) a 128-wide stage of 4 MMAs
// (256 tensor cycles) cannot hide: 2 atoms for 128-wide tiles (+15 % for
// the pair), 1 for 256-wide ones (2 would leave 3 stages or fewer).  Other
// spans use one 128-byte row per stage.
constexpr int stage_atoms(int bn) { return bn == 128 ? 2 : 1; }
constexpr int kThreads = 192;  // 6 warps
constexpr int kSmemBudget = 200 * 1024;
constexpr int kSchedDepth = 4;            // slots of the dynamic scheduler's ring
constexpr uint32_t kNoWork = 0xFFFFFFFFu;  // ring entry: no more work

template <int BN, bool PAIR, int KA = 1>
struct Cfg {
  static constexpr int CG = PAIR ? 2 : 1;
  static constexpr int BN_LOCAL = PAIR ? BN / 2 : BN;  // B columns this CTA loads
  static constexpr int A_BYTES = BM * 128 * KA;        // 128 rows of KA 128-byte atoms
  static constexpr int B_BYTES = 128 * KA * BN_LOCAL;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = kSmemBudget / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int UMMA_M = PAIR ? 256 : 128;
  static constexpr uint32_t TX_BYTES = uint32_t(CG) * STAGE_BYTES;
  // epilogue staging: per epilogue warp two 32 x 32 fp32 boxes (128-byte
  // rows, 128-byte swizzle), written from registers and stored by TMA
  static constexpr int STG_BOX_BYTES = 32 * 32 * 4;
  static constexpr int STG_BYTES = 4 * 2 * STG_BOX_BYTES;
  // stage full/empty, accumulator full/empty, drain, scheduler ring
  // full/empty barriers; TMEM address, abort flag; the ring's work indices
  static constexpr int BAR_BYTES = (2 * STAGES + 5 + 2 * kSchedDepth) * 8 + 8 + 4 * kSchedDepth;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + BAR_BYTES;
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte swizzle atoms");
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation size");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Instruction descriptor of tcgen05.mma kind::f16 / kind::tf32: D fp32
// (bits 4-5 = 1), A and B format (bits 7-9, 10-12: 0 fp16, 1 bf16, 2 tf32 --
// the swz_dtype values), A K-major (bit 15 = 0), B MN-major (bit 16 = 1) or
// K-major (0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int dtype, int m, int n, bool b_mn_major) {
  return (1u << 4) | (uint32_t(dtype) << 7) | (uint32_t(dtype) << 10) |
         (uint32_t(b_mn_major ? 1 : 0) << 16) | (uint32_t(n >> 3) << 17) |
         (uint32_t(m >> 4) << 24);
}

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29), stride byte offset >> 4 (32-45), the fixed
// 0b001 at bits 46-48, base offset 0 (atoms are aligned to their size), and
// the layout type at bits 61-63: 2 = 128-byte swizzle, 4 = 64-byte, 6 =
// 32-byte.
__host__ __device__ constexpr uint32_t sw_layout_type(uint32_t span) {
  return span == 128 ? 2u : span == 64 ? 4u : 6u;
}
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t layout) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
         (uint64_t(layout) << 61);
}

struct Params {
  float* C;
  int M, N, K;
  int order, group;
  uint32_t sched_m, sched_n;  // scheduler grid (cluster tiles with PAIR)
  uint32_t num_kb;            // ceil(K / BK)
  uint32_t idesc;       // MMA instruction descriptor (N = BN)
  uint32_t b3d;         // B's share of a full-width tile in one 3-D box (N % span == 0)
  uint32_t b_kmajor;    // B given as N x K (K contiguous): K-major operand
  uint32_t a3d;         // A's stage in one 3-D box (span < 128 and K % span == 0)
  int32_t* trace;
  uint32_t debug_flags;
  uint64_t timeout_ns;
  // tail policy (persistent launches only; 0 = whole tiles everywhere)
  uint32_t stream_k;
  uint32_t epoch;      // value a finished partial's flag takes in this launch
  uint32_t* sk_flags;  // [cluster][rank][lane quarter]
  float4* sk_ws;       // [cluster][rank][BN/4 column groups][128 rows] float4
  uint32_t* dyn_counter;  // dynamic scheduler: work indices claimed beyond the first wave
  uint32_t epi_pace_ns;   // gap between an epilogue warp's chunk stores (tiles with a successor)
  // die split (static schedules): cluster g sits on die cl_info[g] >> 15 with
  // rank cl_info[g] & 0x7FFF among that die's clusters; die 0's P0 clusters
  // take the units [0, U0) of the tile order, die 1's the rest
  uint32_t die_split, P0, U0;
  uint16_t cl_info[256];
};

enum ItemKind : int { kWhole = 0, kFirst = 1, kPartial = 2 };

// The work of one cluster.  Scheduler units (output tiles, cluster tiles in a
// pair) are the tile order applied to work index w; whole tiles are dealt out
// statically, w = cluster, cluster + P, ... (the persistent loop of the first
// page, work_idx striding of the cluster scheduler).  With stream_k, only the
// first floor(U/P)*P units go out whole; the K iterations of the R = U mod P
// tail units are laid end to end (R*kb iterations) and split into P
// contiguous ranges, one per cluster, so the last wave is shared by every
// cluster instead of running on R of them.  A range is shorter than one tile
// (R < P), so it holds at most two pieces: one in the tile where it starts
// and the head of the next tile.  The pieces of a tile are added in K order
// and the sum written to C by the tile's participants together, each taking
// a share of its chunks (the epilogue).
// Quotient and remainder of 64-bit operands that nearly always fit in 32
// bits: a 32-bit division is a short inline sequence, a 64-bit one a
// subroutine of a few hundred cycles, and the schedule's arithmetic runs
// before the first load is issued.
__device__ __forceinline__ uint64_t div_u64(uint64_t a, uint64_t b) {
  return ((a | b) >> 32) == 0 ? uint64_t(uint32_t(a) / uint32_t(b)) : a / b;
}
__device__ __forceinline__ uint64_t mod_u64(uint64_t a, uint64_t b) {
  return ((a | b) >> 32) == 0 ? uint64_t(uint32_t(a) % uint32_t(b)) : a % b;
}

struct Schedule {
  uint32_t c, P, U, kb;
  uint32_t dp_end;    // units below this are whole tiles
  uint32_t n_dp;      // whole tiles of this cluster
  uint32_t n_pieces;  // tail tiles this cluster's range touches (0, 1 or 2)
  uint32_t ubase;     // the units of this schedule are ubase .. ubase + U - 1 of the order
  uint32_t wsbase;    // first Stream-K workspace cluster slot of this schedule's clusters
  uint64_t I;       // Stream-K tail iterations
  uint64_t s, e;    // this cluster's Stream-K tail range [s, e)
  uint64_t Iq;      // I / P and I % P: range starts are stepped from one
  uint32_t Ir;      // cluster to the next by addition (64-bit division is slow)

  __device__ __forceinline__ void init(uint32_t c_, uint32_t P_, uint32_t U_, uint32_t kb_,
                                       bool sk) {
    c = c_;
    P = P_;
    U = U_;
    kb = kb_;
    ubase = 0;
    wsbase = 0;
    const uint32_t R = sk ? U % P : 0u;
    dp_end = U - R;
    n_dp = c < dp_end ? (dp_end - c + P - 1) / P : 0u;
    I = uint64_t(R) * kb;
    s = e = Iq = 0;
    Ir = 0;
    n_pieces = 0;
    if (I == 0) return;  // whole tiles only
    s = range_start(c);
    e = range_start(c + 1);
    n_pieces = s < e ? uint32_t(div_u64(e - 1, kb) - div_u64(s, kb) + 1) : 0u;
    Iq = div_u64(I, P);
    Ir = uint32_t(mod_u64(I, P));
  }
  __device__ __forceinline__ uint64_t range_start(uint32_t cc) const {
    return div_u64(I * cc, P);
  }
  // Walks the range starts of clusters cc, cc + 1, ...: s = range_start(cc),
  // r = (I * cc) mod P, so that range_start(cc + 1) = s + Iq + carry.
  struct Cursor {
    uint64_t s;
    uint32_t r, cc;
  };
  __device__ __forceinline__ Cursor cursor(uint32_t cc) const {
    const uint64_t t = I * cc;
    return Cursor{div_u64(t, P), uint32_t(mod_u64(t, P)), cc};
  }
  __device__ __forceinline__ void step(Cursor& k) const {
    k.s += Iq;
    k.r += Ir;
    if (k.r >= P) {
      k.r -= P;
      ++k.s;
    }
    ++k.cc;
  }
  // Participants of tail tile t (the clusters whose non-empty ranges meet
  // its K blocks [t*kb, (t+1)*kb)), walked in K order with a cursor:
  // first_part(t) is the cluster holding the tile's first block, and
  // next_part moves to the next cluster with a non-empty range starting
  // before `end` (cc = P when there is none).  A participant's piece of the
  // tile sits in its workspace slot 1 when its range started in an earlier
  // tile (the piece is the head of t), else in slot 0.
  __device__ __forceinline__ uint32_t holder(uint64_t x) const {
    return uint32_t(div_u64((x + 1) * P - 1, I));  // largest cc with range_start(cc) <= x
  }
  __device__ __forceinline__ Cursor first_part(uint32_t t) const {
    return cursor(holder(uint64_t(t) * kb));
  }
  __device__ __forceinline__ void next_part(Cursor& k, uint64_t end) const {
    for (;;) {
      step(k);
      if (k.cc >= P || k.s >= end) {
        k.cc = P;
        return;
      }
      Cursor kn = k;
      step(kn);
      if (kn.s > k.s) return;  // non-empty range
    }
  }
  // Tail tile t: its participants (n), how many of them reduce it (nred)
  // and this cluster's index among the participants (j).  The reducers are
  // the first nred participants: all of them, except the last one when its
  // range runs on into tile t + 1 -- that cluster holds the head of t + 1
  // and reduces that tile instead, so that every cluster reduces one tile.
  struct Part {
    uint32_t n, nred, j;
  };
  __device__ __forceinline__ Part participants(uint32_t t) const {
    const uint64_t end = uint64_t(t + 1) * kb;
    Part r{0u, 0u, 0u};
    uint32_t last = 0;
    for (Cursor k = first_part(t); k.cc < P; next_part(k, end)) {
      if (k.cc == c) r.j = r.n;
      last = k.cc;
      ++r.n;
    }
    const bool last_goes_on = t + 1 < U - dp_end && holder(end) == last;
    r.nred = r.n - (last_goes_on && r.n > 1 ? 1u : 0u);
    return r;
  }
  // The i-th piece of work: unit, K-block range [k0, k1) and kind.  The
  // pieces of the tail range come first (in K order), then the whole units:
  // every cluster starts the tail at once, and the reduction of the split
  // tiles runs in the epilogue warps while the MMAs of the whole units go on.
  __device__ __forceinline__ bool item(uint32_t i, uint32_t& unit, uint32_t& k0, uint32_t& k1,
                                       int& kind) const {
    if (i < n_pieces) {
      const uint64_t t = div_u64(s, kb) + i;
      const uint64_t t0 = t * kb;
      const uint32_t a = s > t0 ? uint32_t(s - t0) : 0u;
      const uint32_t b = e < t0 + kb ? uint32_t(e - t0) : kb;
      unit = ubase + dp_end + uint32_t(t);
      k0 = a;
      k1 = b;
      kind = a > 0 ? kPartial : (b == kb ? kWhole : kFirst);
      return true;
    }
    i -= n_pieces;
    if (i >= n_dp) return false;
    unit = ubase + c + i * P;
    k0 = 0;
    k1 = kb;
    kind = kWhole;
    return true;
  }
};

struct Ctl {
  volatile int* abort_flag;
  uint32_t peer_abort[3];  // shared::cluster addresses of the other CTAs' flags
  uint32_t n_peers;        // other CTAs in the cluster
  uint64_t timeout_ns;
};

__device__ __noinline__ void raise_abort(const Ctl& c) {
  atomicCAS(&g_status_word, 0u, 1u);
  *c.abort_flag = 1;
  for (uint32_t j = 0; j < c.n_peers; ++j)
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(c.peer_abort[j]), "r"(1) : "memory");
}

// The waiting part of wait(), out of line: the issuing threads' unrolled
// loops then carry one test and one call per stage instead of a copy of this
// loop each.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Ctl& c) {
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*c.abort_flag) return false;
      if (ptx::global_timer_ns() - t0 > c.timeout_ns) {
        raise_abort(c);
        return false;
      }
    }
  }
}

// Waits for the phase of `bar` with parity `parity`; false if the kernel
// is aborting or the bound expired (then the abort is raised).
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c);
}

// Waits until the 32-bit flag at `flag` (global) equals `value`, with the
// same bound and abort rules as wait().
__device__ __noinline__ bool wait_flag(const uint32_t* flag, uint32_t value, const Ctl& c) {
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 0;; ++n) {
    if (ptx::ld_acquire_gpu(flag) == value) return true;
    if ((n & 15u) == 15u) {
      if (*c.abort_flag) return false;
      if (ptx::global_timer_ns() - t0 > c.timeout_ns) {
        raise_abort(c);
        return false;
      }
      __nanosleep(64);
    }
  }
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = ptx::global_timer_ns();
  while (ptx::global_timer_ns() - t0 < ns) __nanosleep(1000);
}

template <int BN, bool PAIR, int KIND, int SW, bool DYN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA3,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB3,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Params p) {
  constexpr int KA = SW == 128 ? stage_atoms(BN) : 1;
  using K_ = Cfg<BN, PAIR, KA>;
  constexpr int CL = K_::CG;  // CTAs per cluster
  constexpr int STAGES = K_::STAGES;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sA = ptx::smem_u32(smem);
  const uint32_t sB = sA + STAGES * K_::A_BYTES;
  const uint32_t sStg = sA + STAGES * K_::STAGE_BYTES;  // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * K_::STAGE_BYTES + K_::STG_BYTES);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto sfull_bar = [&](uint32_t s) { return bar0 + 8u * (2 * STAGES + 5 + s); };
  auto sempty_bar = [&](uint32_t s) { return bar0 + 8u * (2 * STAGES + 5 + kSchedDepth + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5 + 2 * kSchedDepth);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile uint32_t* ring_w = tmem_slot + 2;

  const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // rank in the CTA pair: which 128 rows of the pair's tile (the leader, rank
  // 0, issues the MMAs)
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    ptx::prefetch_tensormap(&tmA);
    if constexpr (SW != 128) {
      if (p.a3d) ptx::prefetch_tensormap(&tmA3);
    }
    ptx::prefetch_tensormap(&tmB);
    if (p.b3d) ptx::prefetch_tensormap(&tmB3);
    ptx::prefetch_tensormap(&tmC);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);  // the leader's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar(a), 1);
      ptx::mbar_init(tempty_bar(a), PAIR ? 8 : 4);
    }
    ptx::mbar_init(drain_bar, 1);
    if constexpr (DYN) {
      // a slot is refilled once every reader has taken it: the MMA issuer
      // and the 4 epilogue warps of the leader, plus (pair) the peer's
      // producer and 4 epilogue warps
      for (uint32_t r = 0; r < uint32_t(kSchedDepth); ++r) {
        ptx::mbar_init(sfull_bar(r), 1);
        ptx::mbar_init(sempty_bar(r), PAIR ? 10 : 5);
      }
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc<CL>(ptx::smem_u32(tmem_slot), K_::TMEM_COLS);
    ptx::tmem_relinquish<CL>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Ctl ctl;
  ctl.abort_flag = abort_flag;
  ctl.n_peers = CL - 1;
  if constexpr (PAIR) ctl.peer_abort[0] = ptx::map_to_rank(ptx::smem_u32(abort_flag), rank ^ 1u);
  ctl.timeout_ns = p.timeout_ns;

  const uint32_t units = p.sched_m * p.sched_n;
  Schedule sch;
  if (p.die_split) {
    // this cluster's die takes its own share of the units (and of the
    // Stream-K workspace), with the clusters of that die only
    const uint32_t info = p.cl_info[blockIdx.x / CL];
    const bool d1 = (info >> 15) != 0;
    const uint32_t P1 = gridDim.x / CL - p.P0;
    sch.init(info & 0x7FFFu, d1 ? P1 : p.P0, d1 ? units - p.U0 : p.U0, p.num_kb,
             p.stream_k != 0);
    sch.ubase = d1 ? p.U0 : 0u;
    sch.wsbase = d1 ? p.P0 : 0u;
  } else {
    sch.init(blockIdx.x / CL, gridDim.x / CL, units, p.num_kb, p.stream_k != 0);
  }
  // Everything above touches no global memory: with programmatic dependent
  // launch it overlaps the end of the previous kernel of the stream.  The
  // operands, C, the Stream-K workspace and the dynamic counter are touched
  // only after that kernel has completed; the next GEMM of the stream may
  // then start its own prologue on SMs this grid leaves free.
  ptx::grid_dep_wait();
  if (threadIdx.x == 0) ptx::grid_dep_launch_dependents();
  bool aborted = false;

  // Dynamic scheduler (DYN): the producer of the leader CTA claims work
  // indices -- its cluster id first, then P + the value of a global counter
  // it increments atomically -- and publishes each in a ring of
  // kSchedDepth shared-memory slots (also written into the peer CTA of a
  // pair); the MMA issuer, the epilogue warps and the peer's producer read
  // the same sequence from the ring.  kNoWork ends it.  Work items are whole
  // tiles.  next_item gives a role's i-th item: the static schedule, or the
  // ring (`fetch`: this thread claims and publishes).
  auto ring_put = [&](uint32_t i, uint32_t w) -> bool {
    const uint32_t slot = i % uint32_t(kSchedDepth);
    if (!wait(sempty_bar(slot), ((i / uint32_t(kSchedDepth)) & 1u) ^ 1u, ctl)) return false;
    ring_w[slot] = w;
    if constexpr (PAIR) {
      const uint32_t rw =
          ptx::map_to_rank(ptx::smem_u32(const_cast<uint32_t*>(ring_w + slot)), 1);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(rw), "r"(w) : "memory");
      ptx::mbar_arrive_cluster(ptx::map_to_rank(sfull_bar(slot), 1));
    }
    ptx::mbar_arrive(sfull_bar(slot));
    return true;
  };
  auto ring_take = [&](uint32_t i, uint32_t& w) -> bool {
    const uint32_t slot = i % uint32_t(kSchedDepth);
    if (!wait(sfull_bar(slot), (i / uint32_t(kSchedDepth)) & 1u, ctl)) return false;
    w = ring_w[slot];
    if (leader) ptx::mbar_arrive(sempty_bar(slot));
    else ptx::mbar_arrive_cluster(ptx::map_to_rank(sempty_bar(slot), 0));
    return true;
  };
  uint32_t dyn_published = 0;  // the claiming producer: items published so far
  bool dyn_ended = false;
  auto next_item = [&](uint32_t i, bool fetch, uint32_t& w, uint32_t& kbeg, uint32_t& kend,
                       int& kind) -> bool {
    if constexpr (!DYN) {
      return sch.item(i, w, kbeg, kend, kind);
    } else {
      kbeg = 0;
      kend = p.num_kb;
      kind = kWhole;
      if (fetch) {
        // Published one item ahead: the peer CTA's producer learns its next
        // tile from the ring, and publishing only when this producer starts
        // that tile's loads delayed the peer's loads, and with them the
        // pair's MMAs, at every tile boundary.  The first item is the
        // cluster's own index, the rest are claimed.
        while (!dyn_ended && dyn_published <= i + 1u) {
          const uint32_t k = dyn_published;
          uint32_t wk = k == 0 ? sch.c : sch.P + atomicAdd(p.dyn_counter, 1u);
          if (wk >= units) wk = kNoWork;
          if (!ring_put(k, wk)) { aborted = true; return false; }
          ++dyn_published;
          dyn_ended = wk == kNoWork;
        }
        w = kNoWork;
        if (i < dyn_published) w = ring_w[i % uint32_t(kSchedDepth)];
      } else if (!ring_take(i, w)) {
        aborted = true;
        return false;
      }
      return w != kNoWork;
    }
  };
  // warp-wide form for the epilogue warps: lane 0 reads the ring
  auto next_item_warp = [&](uint32_t i, uint32_t& w, uint32_t& kbeg, uint32_t& kend,
                            int& kind) -> bool {
    if constexpr (!DYN) {
      return sch.item(i, w, kbeg, kend, kind);
    } else {
      uint32_t wl = 0;
      int ok = 1;
      if (lane == 0) ok = ring_take(i, wl) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      w = __shfl_sync(0xFFFFFFFFu, wl, 0);
      kbeg = 0;
      kend = p.num_kb;
      kind = kWhole;
      if (!ok) { aborted = true; return false; }
      return w != kNoWork;
    }
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool skip = (p.debug_flags & SWZ_DEBUG_SKIP_FIRST_LOAD) != 0;
      // operand tiles are read again by other CTAs from L2: kept longer than
      // the C lines the epilogues write (+1 to +2 % where A and B fit in L2)
      const uint64_t pol = ptx::l2_policy_evict_last();
      uint32_t w, kbeg, kend;
      int kind;
      // Swizzle span sw: a stage's 128-byte rows are split into 128/sw
      // column groups of sw bytes (xe elements), each a TMA box of its own
      // (or one 3-D box for all of them); a group holds all rows of the
      // operand block, so group g of a K-major block of R rows starts at
      // g * R * sw.  B given as K x N: boxes of xn columns x BK K rows.
      // The span is a template parameter: the 128-byte kernel carries none
      // of the other spans' code (its issuing threads are latency-critical).
      constexpr uint32_t sw = uint32_t(SW);
      const int groups = int(128u / sw);
      const int xe = int(sw) / (KIND == 0 ? 2 : 4);
      const int xn = int(sw) / 2;
      const uint32_t b_box_bytes = uint32_t(BK) * sw;
      const uint32_t n_clusters = gridDim.x / CL;
      for (uint32_t i = 0; !aborted && next_item(i, leader, w, kbeg, kend, kind); ++i) {
        const TileCoord t = tile_of(p.order, w, p.sched_m, p.sched_n, uint32_t(p.group));
        // K ping-pong: the whole tiles of every other wave (w / P odd) take
        // their K blocks in descending order, so that a wave starts on the
        // K slices of the operand panels the previous wave read last, while
        // they are still in L2.  The direction is a function of the tile,
        // not of the cluster, so every scheduler gives a tile the same sums.
        const bool desc = kind == kWhole && ((w / n_clusters) & 1u) != 0;
        const int32_t m0 = int32_t((t.m * CL + rank) * BM);
        // B columns this CTA loads: its share of the tile
        constexpr int local = K_::BN_LOCAL;
        const int32_t n0 = int32_t(t.n * BN + rank * local);
        constexpr int boxes = local / xn;  // xn = 64 when sw == 128
        constexpr uint32_t tx = K_::TX_BYTES;
        for (uint32_t kb = kbeg; kb < kend; ++kb) {
          if (!wait(empty_bar(stage), phase ^ 1u, ctl)) { aborted = true; break; }
          if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), tx);
          if (skip) {
            skip = false;
          } else {
            const uint32_t fb = PAIR ? ptx::map_to_rank(full_bar(stage), 0) : full_bar(stage);
            const uint32_t kq = desc ? kend - 1u - (kb - kbeg) : kb;
            const int32_t k0 = int32_t(kq * bk_elems<KIND>() * KA);
            const uint32_t a_dst = sA + stage * K_::A_BYTES, b_dst = sB + stage * K_::B_BYTES;
            // A: one box of 128 rows per column group, or one 3-D box
            // (xe elements x 128 rows x groups) when the map allows it.
            // B, N-major (K x N given): one 3-D box (xn columns x BK K rows x
            // `boxes` column groups) when the map allows it, else one 2-D box
            // per group; the shared-memory layout is the same either way.
            // B, K-major (N x K given): per column group one 2-D box of
            // `local` rows.
            const bool one_box = p.b3d != 0;
            if constexpr (SW == 128) {
              // K-major operands: one box per 128-byte atom (KA of them);
              // N-major B: boxes of 64 columns x BK * KA rows
              constexpr int ke = bk_elems<KIND>();
              if constexpr (PAIR) {
#pragma unroll
                for (int g = 0; g < KA; ++g)
                  ptx::tma_load_2d_pair(a_dst + g * (BM * 128), &tmA, fb, k0 + g * ke, m0, pol);
                if (p.b_kmajor)
#pragma unroll
                  for (int g = 0; g < KA; ++g)
                    ptx::tma_load_2d_pair(b_dst + g * local * 128, &tmB, fb, k0 + g * ke, n0, pol);
                else if (one_box)
                  ptx::tma_load_3d_pair(b_dst, &tmB3, fb, 0, k0, n0 / 64, pol);
                else
                  for (int j = 0; j < boxes; ++j)
                    ptx::tma_load_2d_pair(b_dst + j * (BK * KA * 128), &tmB, fb, n0 + 64 * j, k0, pol);
              } else {
#pragma unroll
                for (int g = 0; g < KA; ++g)
                  ptx::tma_load_2d(a_dst + g * (BM * 128), &tmA, fb, k0 + g * ke, m0, pol);
                if (p.b_kmajor)
#pragma unroll
                  for (int g = 0; g < KA; ++g)
                    ptx::tma_load_2d(b_dst + g * local * 128, &tmB, fb, k0 + g * ke, n0, pol);
                else if (one_box)
                  ptx::tma_load_3d(b_dst, &tmB3, fb, 0, k0, n0 / 64, pol);
                else
                  for (int j = 0; j < boxes; ++j)
                    ptx::tma_load_2d(b_dst + j * (BK * KA * 128), &tmB, fb, n0 + 64 * j, k0, pol);
              }
            } else if constexpr (PAIR) {
              if (p.a3d)
                ptx::tma_load_3d_pair(a_dst, &tmA3, fb, 0, m0, k0 / xe, pol);
              else
                for (int g = 0; g < groups; ++g)
                  ptx::tma_load_2d_pair(a_dst + g * BM * sw, &tmA, fb, k0 + g * xe, m0, pol);
              if (p.b_kmajor)
                for (int g = 0; g < groups; ++g)
                  ptx::tma_load_2d_pair(b_dst + g * local * sw, &tmB, fb, k0 + g * xe, n0, pol);
              else if (one_box)
                ptx::tma_load_3d_pair(b_dst, &tmB3, fb, 0, k0, n0 / xn, pol);
              else
                for (int j = 0; j < boxes; ++j)
                  ptx::tma_load_2d_pair(b_dst + j * b_box_bytes, &tmB, fb, n0 + xn * j, k0, pol);
            } else {
              if (p.a3d)
                ptx::tma_load_3d(a_dst, &tmA3, fb, 0, m0, k0 / xe, pol);
              else
                for (int g = 0; g < groups; ++g)
                  ptx::tma_load_2d(a_dst + g * BM * sw, &tmA, fb, k0 + g * xe, m0, pol);
              if (p.b_kmajor)
                for (int g = 0; g < groups; ++g)
                  ptx::tma_load_2d(b_dst + g * local * sw, &tmB, fb, k0 + g * xe, n0, pol);
              else if (one_box)
                ptx::tma_load_3d(b_dst, &tmB3, fb, 0, k0, n0 / xn, pol);
              else
                for (int j = 0; j < boxes; ++j)
                  ptx::tma_load_2d(b_dst + j * b_box_bytes, &tmB, fb, n0 + xn * j, k0, pol);
            }
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Tail: wait until every stage has been released, so that no MMA
      // commit (possibly multicast from the leader) is still in flight
      // towards this CTA's barriers when it exits.
      for (int i = 0; i < STAGES && !aborted; ++i) {
        if (!wait(empty_bar(stage), phase ^ 1u, ctl)) aborted = true;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (aborted) spin_ns(50000);  // let copies already issued land
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA) ----------------
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool issued = false;
      uint32_t w, kbeg, kend;
      int kind;
      // Operand layouts of a stage for swizzle span sw (see the producer).
      // K-major block of R rows: 8-row groups 8*sw bytes apart (stride byte
      // offset); MMA k-slice kk (32 bytes of each row) starts at column
      // group kk*32/sw, byte (kk*32) % sw of the row: offset
      // (kk*32/sw)*R*sw + (kk*32)%sw.  N-major B: boxes of xn columns
      // BK*sw bytes apart along N (leading byte offset), 8 K-rows 8*sw apart
      // (stride byte offset); slice kk starts 16 K-rows = 16*sw bytes in.
      // Offsets are in the descriptor's 16-byte units; the address field
      // cannot carry: shared addresses are below 2^18 bytes.
      constexpr uint32_t sw = uint32_t(SW);
      constexpr uint32_t lay = sw_layout_type(sw);
      auto kmajor_off = [&](int kk, uint32_t rows) {
        return uint64_t(((uint32_t(kk) * 32u / sw) * rows * sw + (uint32_t(kk) * 32u) % sw) >> 4);
      };
      const uint32_t idesc = p.idesc;
      const bool bkm = p.b_kmajor != 0;
      constexpr uint32_t b_rows = uint32_t(K_::BN_LOCAL);
      // 128-byte span: the descriptors of stage 0, built once; stage st's
      // are these plus its offset in 16-byte units (the address field cannot
      // carry).  Building them per stage from the stage address, with the B
      // layout re-read from the parameters after every MMA (whose asm
      // clobbers memory), cost the 128-wide tiles, whose issuing thread is
      // their bound, 1.4-2.5 %.
      const uint64_t adesc0 = make_sdesc(sA, 16, 1024, 2);
      const uint64_t bdesc0 =
          bkm ? make_sdesc(sB, 16, 1024, 2) : make_sdesc(sB, BK * KA * 128, 1024, 2);
      for (uint32_t i = 0; !aborted && next_item(i, false, w, kbeg, kend, kind); ++i) {
        if (!wait(tempty_bar(acc), acc_phase ^ 1u, ctl)) { aborted = true; break; }
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        uint64_t a_step[4] = {}, b_step[4] = {};
        if constexpr (SW != 128) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            a_step[kk] = kmajor_off(kk, BM);
            b_step[kk] = bkm ? kmajor_off(kk, b_rows) : uint64_t((16u * sw * kk) >> 4);
          }
        }
        // One stage's MMAs (4 * KA k-slices of 16 / 8 elements) and the
        // commit that releases the stage when they complete.
        auto issue_stage = [&](uint32_t st, bool first) {
          if constexpr (SW == 128) {
            // slice kk of the KA atoms: atom kk / 4, 32 bytes per slice
            // inside it; N-major B: 16 K-rows of 128 bytes per slice
            const uint64_t adesc = adesc0 + uint64_t(st * uint32_t(K_::A_BYTES >> 4));
            const uint64_t bdesc = bdesc0 + uint64_t(st * uint32_t(K_::B_BYTES >> 4));
            const uint32_t b_atom = b_rows * 128u;  // K-major B: bytes of one atom
            const uint32_t alo = uint32_t(adesc), ahi = uint32_t(adesc >> 32);
            const uint32_t blo = uint32_t(bdesc), bhi = uint32_t(bdesc >> 32);
            ptx::mma<CL, KIND>(d, alo, ahi, blo, bhi, idesc, first ? 0u : 1u);
#pragma unroll
            for (int kk = 1; kk < 4 * KA; ++kk) {
              const uint32_t ao = uint32_t(((kk / 4) * (BM * 128) + (kk % 4) * 32) >> 4);
              const uint32_t bo = bkm ? uint32_t(((kk / 4) * b_atom + (kk % 4) * 32u) >> 4)
                                      : uint32_t(128 * kk);
              ptx::mma<CL, KIND>(d, alo + ao, ahi, blo + bo, bhi, idesc, 1u);
            }
          } else {
            const uint32_t a_addr = sA + st * K_::A_BYTES;
            const uint32_t b_addr = sB + st * K_::B_BYTES;
            const uint64_t adesc = make_sdesc(a_addr, 16, 8 * sw, lay);
            const uint64_t bdesc = bkm ? make_sdesc(b_addr, 16, 8 * sw, lay)
                                       : make_sdesc(b_addr, BK * sw, 8 * sw, lay);
            ptx::mma<CL, KIND>(d, adesc, bdesc, idesc, first ? 0u : 1u);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk)
              ptx::mma<CL, KIND>(d, adesc + a_step[kk], bdesc + b_step[kk], idesc, 1u);
          }
          issued = true;
          // the stage is free (in both CTAs of a pair) once these MMAs are done
          if constexpr (PAIR) ptx::mma_commit_pair(empty_bar(st), 0x3);
          else ptx::mma_commit(empty_bar(st));
        };
        // The issuing thread is the critical path: an MMA takes nearly as
        // long to issue as a 128-wide one takes to run (64 tensor cycles),
        // and every barrier test and branch between MMAs leaves the tensor
        // pipe idle, so the k-loop is unrolled and the barrier test that
        // usually succeeds is the non-blocking one.  (Taking the two-atom
        // stages two at a time, 16 MMAs per test, was slower: a stage then
        // waits for its successor's data too, which halves the time the
        // producer has to refill every other stage.)
#pragma unroll 8
        for (uint32_t kb = kbeg; kb < kend; ++kb) {
          if (!wait(full_bar(stage), phase, ctl)) { aborted = true; break; }
          ptx::tc_fence_after();
          issue_stage(stage, kb == kbeg);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (aborted) break;
        if constexpr (PAIR) ptx::mma_commit_pair(tfull_bar(acc), 0x3);
        else ptx::mma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (aborted && issued) {
        // drain: wait (bounded) until every MMA issued so far has completed
        if constexpr (PAIR) ptx::mma_commit_pair(drain_bar, 0x1);
        else ptx::mma_commit(drain_bar);
        const uint64_t t0 = ptx::global_timer_ns();
        while (!ptx::mbar_try_wait(drain_bar, 0) && ptx::global_timer_ns() - t0 < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: TMEM -> registers -> C ----------------
    // Warp w owns TMEM lanes (rows) 32*(w%4) .. +31 of the accumulator, in
    // chunks of 32 columns.  A whole tile goes to C chunk by chunk.  A piece
    // of a split Stream-K tile (the cluster's first items) is published
    // instead: all its chunks go to this cluster's workspace slot, released
    // per warp with a flag, and the accumulator is freed at once.  After its
    // last piece, the warp reduces its share of the split tiles this cluster
    // reduces -- every piece of a chunk added in K order -- and writes that
    // share of C, while the MMA warp already works on the whole tiles.  So
    // the partial sums of a split tile are spread over its participants, and
    // their exchange overlaps the rest of the launch.
    constexpr uint32_t NCH = uint32_t(BN / 32);  // chunks per warp and tile
    const uint32_t q = warp & 3u;
    uint32_t acc = 0, acc_phase = 0;
    uint32_t w, kbeg, kend;
    int kind;
    const uint32_t stg_warp = sStg + (warp - 2u) * 2u * K_::STG_BOX_BYTES;
    uint32_t nstored = 0;  // chunks stored so far (they alternate between two boxes)
    const uint64_t cpol = ptx::l2_policy_evict_first();  // C is written once
    // One 32 x 32 chunk: registers -> staging box (row r at r*128 bytes, its
    // 16-byte piece j at slot j ^ (r mod 8): the 8 lanes of each 16-byte
    // phase hit 8 different bank groups) -> TMA store at C (col, row), parts
    // beyond M or N clipped by the tensor map.
    auto store_chunk = [&](float (&f)[32], int32_t col, int32_t row) {
      const uint32_t box = stg_warp + (nstored & 1u) * K_::STG_BOX_BYTES;
      ++nstored;
      // the store that last read this box (two chunks ago) must be done
      if (lane == 0) ptx::bulk_wait_group_read<1>();
      __syncwarp();
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t dst = box + lane * 128u + ((uint32_t(v) ^ (lane & 7u)) << 4);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(f[4 * v]),
                     "f"(f[4 * v + 1]), "f"(f[4 * v + 2]), "f"(f[4 * v + 3])
                     : "memory");
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(&tmC, box, col, row, cpol);
        ptx::bulk_commit_group();
      }
    };
    // Stream-K workspace: per cluster two slots (its range's piece in the
    // tile where the range starts, and the head of the next tile), per slot
    // and CTA of the cluster one 4 KB block per warp and chunk (float4 of
    // column group v and row r at v*32 + r) and one flag per warp.
    auto sk_flag = [&](uint32_t cc, uint32_t slot) {
      return p.sk_flags + (((sch.wsbase + cc) * 2u + slot) * uint32_t(CL) + rank) * 4u + q;
    };
    auto sk_block = [&](uint32_t cc, uint32_t slot, uint32_t ch) {
      return p.sk_ws + ((size_t((sch.wsbase + cc) * 2u + slot) * CL + rank) * 4u + q) * (NCH * 256u) +
             size_t(ch) * 256u;
    };
    // Reduces this warp's share of split tile `unit` (nothing if this
    // cluster is not one of its reducers): chunk (q, ch) of a tile with nred
    // reducers belongs to participant (q * NCH + ch) mod nred.  Waits for the
    // participants' flags, then adds their blocks of each chunk in K order
    // and stores the sum.
    auto reduce_tile = [&](uint32_t unit) -> bool {
      const uint32_t tt = unit - sch.ubase - sch.dp_end;
      const uint64_t t_beg = uint64_t(tt) * sch.kb, t_end = t_beg + sch.kb;
      const Schedule::Part pt = sch.participants(tt);
      if (pt.j >= pt.nred) return true;  // not a reducer of this tile
      const uint32_t ch0 = (pt.j + pt.nred - (q * NCH) % pt.nred) % pt.nred;
      if (ch0 >= NCH) return true;  // no chunk of this warp
      bool got = true;
      if (lane == 0) {
        for (Schedule::Cursor k = sch.first_part(tt); k.cc < sch.P; sch.next_part(k, t_end))
          if (!wait_flag(sk_flag(k.cc, k.s < t_beg ? 1u : 0u), p.epoch, ctl)) {
            got = false;
            break;
          }
      }
      if (__shfl_sync(0xFFFFFFFFu, got ? 1 : 0, 0) == 0) return false;
      __threadfence();  // the acquired partial sums before this warp's loads of them
      const TileCoord tc = tile_of(p.order, unit, p.sched_m, p.sched_n, uint32_t(p.group));
      const int32_t row0 = int32_t((tc.m * CL + rank) * BM + q * 32u);
      const int32_t col0 = int32_t(tc.n) * BN;
#pragma unroll 1
      for (uint32_t ch = ch0; ch < NCH; ch += pt.nred) {
        float f[32];
        bool first = true;
        for (Schedule::Cursor k = sch.first_part(tt); k.cc < sch.P; sch.next_part(k, t_end)) {
          const float4* bx = sk_block(k.cc, k.s < t_beg ? 1u : 0u, ch);
          float4 x[8];
#pragma unroll
          for (int v = 0; v < 8; ++v) x[v] = __ldcg(bx + v * 32 + lane);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            f[4 * v] = first ? x[v].x : f[4 * v] + x[v].x;
            f[4 * v + 1] = first ? x[v].y : f[4 * v + 1] + x[v].y;
            f[4 * v + 2] = first ? x[v].z : f[4 * v + 2] + x[v].z;
            f[4 * v + 3] = first ? x[v].w : f[4 * v + 3] + x[v].w;
          }
          first = false;
        }
        store_chunk(f, col0 + int32_t(ch * 32u), row0);
      }
      return true;
    };
    for (uint32_t i = 0; next_item_warp(i, w, kbeg, kend, kind); ++i) {
      const bool ok = wait(tfull_bar(acc), acc_phase, ctl);
      if (!__all_sync(0xFFFFFFFFu, ok)) { aborted = true; break; }
      ptx::tc_fence_after();
      const TileCoord t = tile_of(p.order, w, p.sched_m, p.sched_n, uint32_t(p.group));
      const uint32_t cta_m = t.m * CL + rank, cta_n = t.n;
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + acc * BN;
      if (kind != kWhole) {
        // a piece of a split tile: publish all its chunks, free the accumulator
        const uint32_t tt = w - sch.ubase - sch.dp_end;
        const uint32_t slot = sch.s < uint64_t(tt) * sch.kb ? 1u : 0u;
#pragma unroll 1
        for (uint32_t ch = 0; ch < NCH; ++ch) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + ch * 32u, r);
          ptx::tmem_ld_wait();
          float4* blk = sk_block(sch.c, slot, ch);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            __stcg(blk + v * 32 + lane,
                   make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                               __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
        }
        ptx::tc_fence_before();
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
          else ptx::mbar_arrive(tempty_bar(acc));
          ptx::st_release_gpu(sk_flag(sch.c, slot), p.epoch);
          // the trace names the cluster holding the tile's first K block
          if (warp == 2 && p.trace && kind == kFirst) {
            const uint64_t idx = uint64_t(cta_m) * p.sched_n + cta_n;
            p.trace[2 * idx] = int32_t(blockIdx.x);
            p.trace[2 * idx + 1] = int32_t(i);
          }
        }
        if (i + 1 == sch.n_pieces) {
          // the last piece: reduce the split tiles (one of them, as a rule)
          bool okr = true;
#pragma unroll 1
          for (uint32_t h = 0; h < sch.n_pieces && okr; ++h) {
            uint32_t wh, bh, eh;
            int kh;
            sch.item(h, wh, bh, eh, kh);
            okr = reduce_tile(wh);
          }
          if (!okr) { aborted = true; break; }
        }
      } else {
        const int32_t row0 = int32_t(cta_m * BM + q * 32u);
        const int32_t col0 = int32_t(cta_n) * BN;
        // A tile's C leaves as 4 x BN/32 TMA stores of 4 KB; issued in one
        // burst they share the TMA unit with the operand loads of the next
        // tile's first stages, and the MMA thread stalls there.  When another
        // tile follows, the stores are spread out with a short gap (about a
        // sixteenth of a tile's duration, set on the host); the last tile's
        // epilogue, which nothing overlaps, goes at full speed.
        uint64_t pace_ns = 0;
        if constexpr (!DYN) {
          uint32_t w2, b2, e2;
          int k2;
          if (p.epi_pace_ns && sch.item(i + 1, w2, b2, e2, k2)) pace_ns = p.epi_pace_ns;
        } else {
          // the ring's next slot, if the producer has published it already
          // (it claims a tile before loading it, so usually long before);
          // only looked at, not taken
          const uint32_t nx = (i + 1) % uint32_t(kSchedDepth);
          if (p.epi_pace_ns &&
              ptx::mbar_test_wait(sfull_bar(nx), ((i + 1) / uint32_t(kSchedDepth)) & 1u) &&
              ring_w[nx] != kNoWork)
            pace_ns = p.epi_pace_ns;
        }
#pragma unroll 1
        for (uint32_t ch = 0; ch < NCH; ++ch) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + ch * 32u, r);
          ptx::tmem_ld_wait();
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
          store_chunk(f, col0 + int32_t(ch * 32u), row0);
          if (pace_ns && ch + 1 < NCH) {
            const uint64_t t0 = ptx::global_timer_ns();
            while (ptx::global_timer_ns() - t0 < pace_ns) __nanosleep(100);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
          else ptx::mbar_arrive(tempty_bar(acc));
          if (warp == 2 && p.trace) {
            const uint64_t idx = uint64_t(cta_m) * p.sched_n + cta_n;
            p.trace[2 * idx] = int32_t(blockIdx.x);
            p.trace[2 * idx + 1] = int32_t(i);
          }
        }
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---------------- teardown ----------------
  if (warp >= 2 && lane == 0) ptx::bulk_wait_group<0>();  // C stores complete
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc<CL>(tmem_base, K_::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// element type of a tensor map: the operands' fp16 / bf16, or fp32 for C
constexpr int kMapF32 = 100;

static CUtensorMapSwizzle tma_swizzle(uint32_t span) {
  return span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                      : CU_TENSOR_MAP_SWIZZLE_32B;
}

static CUtensorMapDataType tma_type(int dtype) {
  // TF32 operands are copied bit for bit (FLOAT32); the tensor core reads
  // them as TF32
  return (dtype == kMapF32 || dtype == SWZ_TF32) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
         : dtype == SWZ_BF16                      ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// 2-D row-major matrix rows x cols, box box_cols x box_rows, swizzle span
// `span` bytes (box_cols * element size must not exceed it); out-of-bounds
// elements read as zero and are not written by stores.
static int encode_2d(CUtensorMap* map, int dtype, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_cols, uint32_t box_rows, uint32_t span = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const uint64_t esize = (dtype == kMapF32 || dtype == SWZ_TF32) ? 4 : 2;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, tma_type(dtype), 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, tma_swizzle(span),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return SWZ_OK;
}

// A row-major rows x cols matrix (cols % gcols == 0) seen as a 3-D tensor
// (gcols columns, rows, cols / gcols column groups); box gcols x box_rows x
// box_groups, swizzle span `span` (= gcols * element size).  In shared
// memory the box is box_groups consecutive box_rows x gcols blocks, the
// layout of box_groups 2-D boxes side by side.  Only for cols % gcols == 0:
// a partial last group would read the next row's elements instead of zeros.
static int encode_groups(CUtensorMap* map, int dtype, const void* base, uint64_t rows,
                         uint64_t cols, uint32_t gcols, uint32_t box_rows, uint32_t box_groups,
                         uint32_t span) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cuda_fail(cudaErrorNotSupported);
  const uint64_t esize = (dtype == kMapF32 || dtype == SWZ_TF32) ? 4 : 2;
  const cuuint64_t dims[3] = {gcols, rows, cols / gcols};
  const cuuint64_t strides[2] = {cols * esize, gcols * esize};
  const cuuint32_t box[3] = {gcols, box_rows, box_groups};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, tma_type(dtype), 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, tma_swizzle(span),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return SWZ_OK;
}

struct Plan {
  int bn;
  bool pair;
  uint32_t tiles_m, tiles_n, sched_m, sched_n, units;
  int programs;
};

template <int BN, bool PAIR, int KIND>
static int kernel_capacity(const DeviceInfo& dev, int* programs) {
  constexpr int SW = 128;
  constexpr int CLN = PAIR ? 2 : 1;
  using K_ = Cfg<BN, PAIR, stage_atoms(BN)>;
  static std::mutex mu;
  static int cache[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev.device] > 0) {
      *programs = cache[dev.device];
      return SWZ_OK;
    }
  }
  auto kern = gemm_kernel<BN, PAIR, KIND, SW, false>;
  SWZ_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    K_::SMEM_BYTES));
  int cap = 0;
  if constexpr (PAIR) {
    // clusters fit a GPC only whole: ask the occupancy API how many can be
    // resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CLN * dev.num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = K_::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLN;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    SWZ_CUDA_TRY(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg));
    cap = CLN * clusters;
  } else {
    int per_sm = 0;
    SWZ_CUDA_TRY(
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, K_::SMEM_BYTES));
    cap = per_sm * dev.num_sms;
  }
  if (cap <= 0) return SWZ_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  cache[dev.device] = cap;
  *programs = cap;
  return SWZ_OK;
}

static int capacity_for(const Plan& pl, const DeviceInfo& dev, int* cap) {
  // the three configurations share their shared-memory footprint across
  // kinds, so the f16 kernels' residency stands for both
  if (pl.pair) {
    if (pl.bn == 128) return kernel_capacity<128, true, 0>(dev, cap);
    return kernel_capacity<256, true, 0>(dev, cap);
  }
  if (pl.bn == 128) return kernel_capacity<128, false, 0>(dev, cap);
  return kernel_capacity<256, false, 0>(dev, cap);
}

static int make_plan(int M, int N, int persistent, const swz_gemm_opts& o, const DeviceInfo* dev,
                     Plan* pl) {
  if (o.tile_n != 0 && o.tile_n != 128 && o.tile_n != 256) return SWZ_EUNSUPPORTED;
  pl->pair = o.cta_pair != 0;
  pl->bn = o.tile_n ? o.tile_n : (pl->pair || N > 128 ? 256 : 128);
  const int cln = pl->pair ? 2 : 1;  // CTAs per cluster (a pair is stacked in M)
  const uint64_t sm = (uint64_t(M) + BM * cln - 1) / (BM * cln);
  const uint64_t sn = (uint64_t(N) + uint64_t(pl->bn) - 1) / uint64_t(pl->bn);
  if (sm * sn * cln > uint64_t(INT32_MAX)) return SWZ_EINVAL;
  pl->sched_m = uint32_t(sm);
  pl->sched_n = uint32_t(sn);
  pl->tiles_m = uint32_t(sm * cln);
  pl->tiles_n = uint32_t(sn);
  pl->units = uint32_t(sm * sn);
  if (o.num_programs < 0 || (o.num_programs % cln) != 0) return SWZ_EINVAL;
  if (!persistent) {
    pl->programs = int(pl->units) * cln;
  } else {
    int cap = o.num_programs;
    if (cap == 0) {
      if (!dev) return SWZ_EINVAL;
      const int rc = capacity_for(*pl, *dev, &cap);
      if (rc != SWZ_OK) return rc;
    }
    const uint32_t units_cap = uint32_t(cap / cln);
    // Stream-K shares the tail among all programs, so with fewer units than
    // programs (the whole product is one partial wave) every program stays
    // and each unit's K iterations are split among several of them.
    pl->programs = int(pl->units < units_cap && !o.stream_k ? pl->units : units_cap) * cln;
  }
  return SWZ_OK;
}

// Stream-K workspace: flags [clusters][2 slots][CL][4 warps] uint32 (a
// 256-byte aligned block), then partial sums [clusters][2 slots][CL][4
// warps][BN/32 chunks] of 4 KB blocks (32 rows x 32 fp32 columns).
struct SkLayout {
  bool active;
  uint64_t flags_bytes, data_bytes;
};

// workspace of a dynamic-scheduler launch: the claimed-work counter
constexpr uint64_t kDynWorkspaceBytes = 256;

static SkLayout sk_layout(const Plan& pl, int persistent, const swz_gemm_opts& o) {
  SkLayout L{false, 0, 0};
  const uint32_t cl = pl.pair ? 2u : 1u;
  const uint32_t clusters = uint32_t(pl.programs) / cl;
  if (!o.stream_k || !persistent || clusters == 0 || pl.units % clusters == 0) return L;
  L.active = true;
  L.flags_bytes = (uint64_t(clusters) * 2u * cl * 4u * 4u + 255u) & ~uint64_t(255);
  L.data_bytes = uint64_t(clusters) * 2u * cl * BM * uint64_t(pl.bn) * 4u;
  return L;
}

// ---- die split ----------------------------------------------------------
// What swz_calibrate found on each device: the die of every SM, and the SM
// of every CTA of each persistent kernel shape (clusters, shared memory,
// CTAs) launched at its resident capacity.
struct DieCalibration {
  bool have = false;
  std::vector<uint8_t> die_of_sm;
  std::map<std::tuple<int, int, int>, std::vector<uint32_t>> placement;
};
static std::mutex g_die_mu;
static DieCalibration g_die_cal[64];

// dynamic shared memory of the kernel a launch of this plan and span uses
static int kernel_smem(const Plan& pl, uint32_t span) {
  const bool ka2 = span == 128 && pl.bn == 128;
  if (pl.pair) {
    if (pl.bn == 256) return Cfg<256, true, 1>::SMEM_BYTES;
    return ka2 ? Cfg<128, true, 2>::SMEM_BYTES : Cfg<128, true, 1>::SMEM_BYTES;
  }
  if (pl.bn == 256) return Cfg<256, false, 1>::SMEM_BYTES;
  return ka2 ? Cfg<128, false, 2>::SMEM_BYTES : Cfg<128, false, 1>::SMEM_BYTES;
}

struct DieSplit {
  bool on;            // both dies have clusters of this launch
  uint32_t P0, U0;    // clusters on die 0, units die 0 takes
  std::vector<uint16_t> info;  // per cluster: die << 15 | rank on that die
};

// The die split of a persistent launch of plan `pl` (span `span`) on
// device `dev`: SWZ_EUNSUPPORTED when the device was not calibrated.  A
// launch whose shape calibration did not place (a program count other than
// the resident capacity) gets no split (ds->on false).
static int die_split_of(const Plan& pl, uint32_t span, int dev, DieSplit* ds) {
  const int cl = pl.pair ? 2 : 1;
  const uint32_t clusters = uint32_t(pl.programs) / uint32_t(cl);
  std::lock_guard<std::mutex> lock(g_die_mu);
  if (dev < 0 || dev >= 64 || !g_die_cal[dev].have) return SWZ_EUNSUPPORTED;
  ds->on = false;
  ds->P0 = clusters;
  ds->U0 = pl.units;
  ds->info.clear();
  const DieCalibration& cal = g_die_cal[dev];
  const auto it = cal.placement.find(std::make_tuple(cl, kernel_smem(pl, span), pl.programs));
  if (it == cal.placement.end() || clusters == 0 || clusters > 256) return SWZ_OK;
  ds->info.assign(clusters, 0);
  uint32_t n[2] = {0, 0};
  for (uint32_t g = 0; g < clusters; ++g) {
    const uint32_t sm = it->second[size_t(g) * cl];
    const uint32_t d = sm < cal.die_of_sm.size() ? cal.die_of_sm[sm] : 0u;
    ds->info[g] = uint16_t((d << 15) | n[d]++);
  }
  ds->on = n[0] > 0 && n[1] > 0;
  ds->P0 = n[0];
  // each die takes units in proportion to its clusters
  ds->U0 = uint32_t((uint64_t(pl.units) * n[0] + clusters / 2) / clusters);
  return SWZ_OK;
}

template <int BN, bool PAIR, int KIND, int SW, bool DYN>
static int launch(const Plan& pl, const CUtensorMap& ta, const CUtensorMap& ta3,
                  const CUtensorMap& tb, const CUtensorMap& tb3, const CUtensorMap& tc,
                  const Params& prm, cudaStream_t stream) {
  using K_ = Cfg<BN, PAIR, SW == 128 ? stage_atoms(BN) : 1>;
  static std::mutex mu;
  static bool attr_set[64] = {};
  auto kern = gemm_kernel<BN, PAIR, KIND, SW, DYN>;
  int dev = 0;
  SWZ_CUDA_TRY(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      SWZ_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        K_::SMEM_BYTES));
      attr_set[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(pl.programs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = K_::SMEM_BYTES;
  cfg.stream = stream;
  // programmatic stream serialisation: the kernel may start while the
  // previous kernel of the stream finishes (it waits for that kernel's
  // completion before its first access to global memory)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (PAIR) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  SWZ_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, ta, ta3, tb, tb3, tc, prm));
  return SWZ_OK;
}

}  // namespace gemm
}  // namespace swz

using namespace swz;
using namespace swz::gemm;

// kernel instance for the plan's tile shape, the operand kind and span SW
template <int SW, bool DYN>
static int dispatch(const Plan& pl, bool tf32, const CUtensorMap& ta, const CUtensorMap& ta3,
                    const CUtensorMap& tb, const CUtensorMap& tb3, const CUtensorMap& tc,
                    const Params& prm, cudaStream_t s) {
  if (tf32) {
    if (pl.pair && pl.bn == 128)
      return launch<128, true, 1, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
    if (pl.pair) return launch<256, true, 1, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
    if (pl.bn == 128) return launch<128, false, 1, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
    return launch<256, false, 1, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
  }
  if (pl.pair && pl.bn == 128)
    return launch<128, true, 0, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
  if (pl.pair) return launch<256, true, 0, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
  if (pl.bn == 128) return launch<128, false, 0, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
  return launch<256, false, 0, SW, DYN>(pl, ta, ta3, tb, tb3, tc, prm, s);
}

static int validate(const void* A, const void* B, const float* C, int M, int N, int K, int order,
                    int group, const swz_gemm_opts& o) {
  if (M < 0 || N < 0 || K < 0) return SWZ_EINVAL;
  if (!order_is_valid(order)) return SWZ_EINVAL;
  if (order_uses_group(order) && group < 1) return SWZ_EINVAL;
  if (o.dtype != SWZ_F16 && o.dtype != SWZ_BF16 && o.dtype != SWZ_TF32) return SWZ_EINVAL;
  if (o.b_layout != SWZ_B_KN && o.b_layout != SWZ_B_NK) return SWZ_EINVAL;
  if (o.smem_swizzle != 0 && o.smem_swizzle != 32 && o.smem_swizzle != 64 &&
      o.smem_swizzle != 128)
    return SWZ_EINVAL;
  if (M == 0 || N == 0) return SWZ_OK;
  if (!C || !aligned16(C) || N % 4 != 0) return SWZ_EINVAL;
  if (K == 0) return SWZ_OK;
  if (!A || !B || !aligned16(A) || !aligned16(B)) return SWZ_EINVAL;
  // rows of A (and of B given as N x K) and of B given as K x N must be
  // multiples of 16 bytes for TMA
  const int per16 = o.dtype == SWZ_TF32 ? 4 : 8;
  if (K % per16 != 0) return SWZ_EINVAL;
  if (o.b_layout == SWZ_B_KN && N % per16 != 0) return SWZ_EINVAL;
  return SWZ_OK;
}

extern "C" int swz_gemm_plan(int M, int N, int K, int persistent, const swz_gemm_opts* opts,
                             int* tiles_m, int* tiles_n, int* sched_m, int* sched_n,
                             int* programs) {
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  if (M <= 0 || N <= 0 || K < 0) return SWZ_EINVAL;
  DeviceInfo dev{};
  const bool need_dev = persistent && o.num_programs == 0;
  if (need_dev) {
    const int rc = current_device(&dev);
    if (rc != SWZ_OK) return rc;
  }
  Plan pl{};
  const int rc = make_plan(M, N, persistent, o, need_dev ? &dev : nullptr, &pl);
  if (rc != SWZ_OK) return rc;
  if (tiles_m) *tiles_m = int(pl.tiles_m);
  if (tiles_n) *tiles_n = int(pl.tiles_n);
  if (sched_m) *sched_m = int(pl.sched_m);
  if (sched_n) *sched_n = int(pl.sched_n);
  if (programs) *programs = pl.programs;
  return SWZ_OK;
}

extern "C" int swz_calibrate(int* h_die_of_sm, int max_sms, int* h_num_sms) {
  DeviceInfo dev{};
  int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  if (max_sms < 0 || (max_sms > 0 && !h_die_of_sm)) return SWZ_EINVAL;
  DieCalibration cal;
  rc = die_of_sms(dev.num_sms, &cal.die_of_sm);
  if (rc != SWZ_OK) return rc;
  // the placement of every persistent kernel shape at its resident capacity
  for (int pair = 0; pair < 2; ++pair)
    for (int bn : {128, 256})
      for (uint32_t span : {128u, 64u}) {
        Plan pl{};
        pl.pair = pair != 0;
        pl.bn = bn;
        int cap = 0;
        rc = capacity_for(pl, dev, &cap);
        if (rc != SWZ_OK) return rc;
        const auto key = std::make_tuple(pair ? 2 : 1, kernel_smem(pl, span), cap);
        if (cal.placement.count(key)) continue;
        std::vector<uint32_t> sm;
        rc = placement(pair ? 2 : 1, kThreads, kernel_smem(pl, span), cap, &sm);
        if (rc != SWZ_OK) return rc;
        cal.placement[key] = sm;
      }
  cal.have = true;
  if (h_num_sms) *h_num_sms = dev.num_sms;
  for (int s = 0; s < max_sms; ++s)
    h_die_of_sm[s] = s < int(cal.die_of_sm.size()) ? cal.die_of_sm[size_t(s)] : 0;
  std::lock_guard<std::mutex> lock(g_die_mu);
  if (dev.device >= 0 && dev.device < 64) g_die_cal[dev.device] = cal;
  return SWZ_OK;
}

extern "C" int swz_gemm_die_plan(int M, int N, int K, const swz_gemm_opts* opts,
                                 int32_t* h_cluster_info, int max_clusters, int* h_clusters,
                                 int* h_P0, int* h_U0) {
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  if (M <= 0 || N <= 0 || K < 0 || max_clusters < 0 || (max_clusters && !h_cluster_info))
    return SWZ_EINVAL;
  DeviceInfo dev{};
  int rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  Plan pl{};
  rc = make_plan(M, N, 1, o, &dev, &pl);
  if (rc != SWZ_OK) return rc;
  DieSplit ds{};
  rc = die_split_of(pl, o.smem_swizzle ? uint32_t(o.smem_swizzle) : 128u, dev.device, &ds);
  if (rc != SWZ_OK) return rc;
  const int clusters = pl.programs / (pl.pair ? 2 : 1);
  if (h_clusters) *h_clusters = clusters;
  if (h_P0) *h_P0 = ds.on ? int(ds.P0) : clusters;
  if (h_U0) *h_U0 = ds.on ? int(ds.U0) : int(pl.units);
  for (int g = 0; g < max_clusters && g < clusters; ++g)
    h_cluster_info[g] = ds.on ? int32_t(ds.info[size_t(g)]) : int32_t(g);
  return SWZ_OK;
}

namespace swz {
int gemm_sk_workspace_split(int M, int N, int K, int persistent, const swz_gemm_opts& o,
                            uint64_t* flag_bytes, uint64_t* total_bytes) {
  *flag_bytes = *total_bytes = 0;
  if (M <= 0 || N <= 0 || K <= 0 || !o.stream_k || !persistent) return SWZ_OK;
  DeviceInfo dev{};
  const bool need_dev = o.num_programs == 0;
  if (need_dev) {
    const int rc = current_device(&dev);
    if (rc != SWZ_OK) return rc;
  }
  Plan pl{};
  const int rc = make_plan(M, N, persistent, o, need_dev ? &dev : nullptr, &pl);
  if (rc != SWZ_OK) return rc;
  const SkLayout L = sk_layout(pl, persistent, o);
  if (L.active) {
    *flag_bytes = L.flags_bytes;
    *total_bytes = L.flags_bytes + L.data_bytes;
  }
  return SWZ_OK;
}
}  // namespace swz

extern "C" int swz_gemm_workspace_size(int M, int N, int K, int persistent,
                                       const swz_gemm_opts* opts, uint64_t* bytes) {
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  if (!bytes || M < 0 || N < 0 || K < 0) return SWZ_EINVAL;
  *bytes = 0;
  if (o.dynamic && !o.stream_k) {
    *bytes = persistent ? kDynWorkspaceBytes : 0;
    return SWZ_OK;
  }
  if (M == 0 || N == 0 || K == 0 || !o.stream_k || !persistent) return SWZ_OK;
  DeviceInfo dev{};
  const bool need_dev = o.num_programs == 0;
  if (need_dev) {
    const int rc = current_device(&dev);
    if (rc != SWZ_OK) return rc;
  }
  Plan pl{};
  const int rc = make_plan(M, N, persistent, o, need_dev ? &dev : nullptr, &pl);
  if (rc != SWZ_OK) return rc;
  const SkLayout L = sk_layout(pl, persistent, o);
  *bytes = L.active ? L.flags_bytes + L.data_bytes : 0;
  return SWZ_OK;
}

namespace swz {
int gemm_ex(const void* A, const void* B, float* C, int M, int N, int K, int order, int group,
            int persistent, const swz_gemm_opts* opts, void* stream, bool clear_sk_flags) {
  swz_gemm_opts o = {};
  if (opts) o = *opts;
  int rc = validate(A, B, C, M, N, K, order, group, o);
  if (rc != SWZ_OK) return rc;
  if (M == 0 || N == 0) return SWZ_OK;
  DeviceInfo dev{};
  rc = current_device(&dev);
  if (rc != SWZ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    SWZ_CUDA_TRY(cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * sizeof(float), s));
    return SWZ_OK;
  }
  Plan pl{};
  rc = make_plan(M, N, persistent, o, &dev, &pl);
  if (rc != SWZ_OK) return rc;
  const uint32_t g = order_uses_group(order) ? uint32_t(group) : 1u;
  if ((order == kMorton || order == kXor) &&
      !order_is_bijective(order, pl.sched_m, pl.sched_n, g))
    return SWZ_ENOTBIJECTIVE;

  // TF32 operands are taken K-major on both sides (B as N x K)
  if (o.dtype == SWZ_TF32 && o.b_layout != SWZ_B_NK) return SWZ_EUNSUPPORTED;
  const bool tf32 = o.dtype == SWZ_TF32;
  const uint32_t span = o.smem_swizzle ? uint32_t(o.smem_swizzle) : 128u;
  const uint32_t esize = tf32 ? 4u : 2u;
  const uint32_t bke = 128u / esize;  // K elements per 128-byte stage row
  const uint32_t xe = span / esize;   // elements per swizzle span
  // 128-byte K atoms per stage of the kernel this launch will use
  const uint32_t ka = span == 128 ? uint32_t(stage_atoms(pl.bn)) : 1u;
  const uint32_t local = uint32_t(pl.pair ? pl.bn / 2 : pl.bn);  // B columns per CTA
  const bool b_kmajor = o.b_layout == SWZ_B_NK;
  CUtensorMap ta, ta3, tb, tb3, tc;
  // A: boxes of xe elements x 128 rows, one per span-wide column group of a
  // stage; with span < 128 and K % xe == 0, all groups in one 3-D box
  rc = encode_2d(&ta, o.dtype, A, uint64_t(M), uint64_t(K), xe, BM, span);
  if (rc != SWZ_OK) return rc;
  const bool a3d = span < 128 && uint32_t(K) % xe == 0;
  ta3 = ta;
  if (a3d) {
    rc = encode_groups(&ta3, o.dtype, A, uint64_t(M), uint64_t(K), xe, BM, 128 / span, span);
    if (rc != SWZ_OK) return rc;
  }
  bool b3d = false;
  if (b_kmajor) {
    // B given as N x K: like A, boxes of `local` rows
    rc = encode_2d(&tb, o.dtype, B, uint64_t(N), uint64_t(K), xe, local, span);
    if (rc != SWZ_OK) return rc;
    tb3 = tb;
  } else {
    const uint32_t xn = span / 2;  // B columns per span (16-bit elements)
    rc = encode_2d(&tb, o.dtype, B, uint64_t(K), uint64_t(N), xn, BK * ka, span);
    if (rc != SWZ_OK) return rc;
    // B as (xn columns, K rows, N/xn column groups): a CTA's whole share of
    // a tile in one box, when N % xn == 0
    b3d = uint32_t(N) % xn == 0;
    tb3 = tb;
    if (b3d) {
      rc = encode_groups(&tb3, o.dtype, B, uint64_t(K), uint64_t(N), xn, BK * ka, local / xn,
                         span);
      if (rc != SWZ_OK) return rc;
    }
  }
  rc = encode_2d(&tc, kMapF32, C, uint64_t(M), uint64_t(N), 32, 32);
  if (rc != SWZ_OK) return rc;

  Params prm{};
  prm.C = C;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.order = order;
  prm.group = int(g);
  prm.sched_m = pl.sched_m;
  prm.sched_n = pl.sched_n;
  prm.num_kb = uint32_t((uint32_t(K) + bke * ka - 1) / (bke * ka));
  prm.idesc = make_idesc(o.dtype, pl.pair ? 256 : 128, pl.bn, !b_kmajor);
  prm.b_kmajor = b_kmajor ? 1u : 0u;
  prm.a3d = a3d ? 1u : 0u;
  if (o.dynamic < 0 || o.dynamic > 1) return SWZ_EINVAL;
  if (o.dynamic) {
    if (!persistent || o.stream_k) return SWZ_EINVAL;
    const uintptr_t ws = reinterpret_cast<uintptr_t>(o.d_workspace);
    if (!ws || (ws & 255u) || o.workspace_bytes < kDynWorkspaceBytes) return SWZ_EINVAL;
    if (span != 128) return SWZ_EUNSUPPORTED;
  }
  prm.trace = o.d_trace;
  prm.debug_flags = o.debug_flags;
  // epilogue store gap: ~1/16 of a tile's duration (proportional to K and the
  // tile width, twice as long for TF32), at most 1 us; persistent launches
  // only (a CTA of a non-persistent launch has no following tile)
  if (persistent) {
    const uint64_t pace = uint64_t(K) * uint64_t(pl.bn) * (tf32 ? 2u : 1u) / 1024u;
    prm.epi_pace_ns = uint32_t(pace < 1000u ? pace : 1000u);
  }
  prm.timeout_ns = uint64_t(o.timeout_ms ? o.timeout_ms : 2000u) * 1000000ull;

  if (o.stream_k) {
    if (!persistent) return SWZ_EINVAL;
    const SkLayout L = sk_layout(pl, persistent, o);
    if (L.active) {
      // pieces of one tile wait on one another: every program must be resident
      int cap = 0;
      rc = capacity_for(pl, dev, &cap);
      if (rc != SWZ_OK) return rc;
      if (pl.programs > cap) return SWZ_EUNSUPPORTED;
      const uintptr_t ws = reinterpret_cast<uintptr_t>(o.d_workspace);
      if (!ws || (ws & 255u) || o.workspace_bytes < L.flags_bytes + L.data_bytes)
        return SWZ_EINVAL;
      static std::atomic<uint32_t> epoch{0};
      uint32_t e = epoch.fetch_add(1) + 1;
      if (e == 0) e = epoch.fetch_add(1) + 1;
      // A captured launch keeps this epoch in every replay, so a replay would
      // find the previous replay's flags already at it: under capture the
      // flags are cleared on the stream before the launch (a memset node that
      // runs in every replay; epochs are never 0).
      cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
      SWZ_CUDA_TRY(cudaStreamIsCapturing(s, &capturing));
      if (capturing != cudaStreamCaptureStatusNone || clear_sk_flags)
        SWZ_CUDA_TRY(cudaMemsetAsync(reinterpret_cast<void*>(ws), 0, size_t(L.flags_bytes), s));
      prm.stream_k = 1;
      prm.epoch = e;
      prm.sk_flags = reinterpret_cast<uint32_t*>(ws);
      prm.sk_ws = reinterpret_cast<float4*>(ws + L.flags_bytes);
    }
  }

  prm.b3d = b3d ? 1u : 0u;
  if (o.die_split) {
    if (o.die_split != 1 || !persistent || o.dynamic) return SWZ_EINVAL;
    DieSplit ds{};
    rc = die_split_of(pl, span, dev.device, &ds);
    if (rc != SWZ_OK) return rc;
    if (ds.on) {
      prm.die_split = 1;
      prm.P0 = ds.P0;
      prm.U0 = ds.U0;
      for (size_t g = 0; g < ds.info.size(); ++g) prm.cl_info[g] = ds.info[g];
    }
  }
  if (o.dynamic) {
    // the counter of claimed work indices starts at zero in every launch
    prm.dyn_counter = static_cast<uint32_t*>(o.d_workspace);
    SWZ_CUDA_TRY(cudaMemsetAsync(prm.dyn_counter, 0, sizeof(uint32_t), s));
    return dispatch<128, true>(pl, tf32, ta, ta3, tb, tb3, tc, prm, s);
  }
  if (span == 64) return dispatch<64, false>(pl, tf32, ta, ta3, tb, tb3, tc, prm, s);
  if (span == 32) return dispatch<32, false>(pl, tf32, ta, ta3, tb, tb3, tc, prm, s);
  return dispatch<128, false>(pl, tf32, ta, ta3, tb, tb3, tc, prm, s);
}
}  // namespace swz

extern "C" int swz_gemm_ex(const void* A, const void* B, float* C, int M, int N, int K, int order,
                           int group, int persistent, const swz_gemm_opts* opts, void* stream) {
  return swz::gemm_ex(A, B, C, M, N, K, order, group, persistent, opts, stream, false);
}

extern "C" int swz_gemm(const void* A, const void* B, float* C, int M, int N, int K, int order,
                        int group, int persistent, void* stream) {
  return swz_gemm_ex(A, B, C, M, N, K, order, group, persistent, nullptr, stream);
}

extern "C" int swz_check_status(void* stream) {
  SWZ_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  unsigned int v = 0;
  SWZ_CUDA_TRY(cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)));
  if (v != 0) {
    const unsigned int zero = 0;
    SWZ_CUDA_TRY(cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)));
    return SWZ_ETIMEOUT;
  }
  return SWZ_OK;
}
