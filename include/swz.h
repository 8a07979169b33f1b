/*
 * swz.h -- C ABI of libswz.so: thread-block-swizzled GEMM, tile maps and a
 * shared-memory-swizzled transpose for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (cited by page title and section):
 *   [TBS] Lei Mao, "CUDA Thread Block Swizzle" -- tile orders (sections
 *         "Linear Swizzle", "Grouped 2D Panel Swizzle", "Morton / Z-order
 *         Swizzle", "Bitwise XOR Swizzle") and the benchmark's masked tiled
 *         GEMM C = A*B with persistent / non-persistent launch.
 *   [SBC] WHC, "CUDA Swizzle & bank conflict" -- section "Matrix Transpose"
 *         (naive, padded and XOR-swizzled shared-memory tiles) and section
 *         "Hopper TMA 的 swizzling" (the 128-byte swizzle the GEMM's operand
 *         staging uses).
 *   [CPS] TVM TIRx docs, "ClusterPersistentScheduler2D" -- group-major and
 *         serpentine orders, work_idx = cluster_id + i * num_clusters, and
 *         the cluster-tile -> CTA-tile split of "Example 2: 2SM GEMM".
 *
 * Conventions for every call:
 *   - Device pointers are caller-owned global memory on the current device;
 *     the library never allocates, frees or retains them.  Host pointers are
 *     named h_* and are only read or written during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no call synchronises except
 *     swz_check_status.
 *   - CUDA graphs: the calls on device buffers (swz_tile_map, swz_gemm,
 *     swz_gemm_ex, swz_gemm_streamk_noalloc, swz_gemm_mma_sync,
 *     swz_transpose, swz_tc_rate, swz_tc_rate_ex) allocate nothing and do
 *     not synchronise, so they may be recorded by stream capture and the
 *     graph replayed.  The host-buffer calls (swz_gemm_host*) work on
 *     streams of the library's own and are not for capture; neither is
 *     swz_check_status, which synchronises.  Make one ordinary call with
 *     the same configuration on the device first: the first call of each
 *     kernel variant sets its shared-memory limit and caches occupancy and
 *     device queries.  What a call clears before its launch (the dynamic
 *     scheduler's counter, Stream-K's piece flags) is recorded as a memset
 *     and cleared again in every replay; a captured call keeps its
 *     arguments, so buffers are rewritten in place between replays.
 *   - Every call returns SWZ_OK (0) or a negative swz_status.  Arguments are
 *     validated before anything is enqueued; on error nothing is enqueued.
 *     No exception crosses the ABI.  Calls are thread-safe; the only
 *     library-global state is the per-device status word read by
 *     swz_check_status and the last CUDA error code.
 */
#ifndef SWZ_H_
#define SWZ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
enum swz_status {
  SWZ_OK = 0,
  SWZ_EINVAL = -1,         /* null pointer, bad size, bad enum, misalignment */
  SWZ_ENOTBIJECTIVE = -2,  /* Morton/XOR order not a permutation of this grid */
  SWZ_EARCH = -3,          /* current device is not sm_103 (GB300)            */
  SWZ_ECUDA = -4,          /* a CUDA runtime call failed: swz_last_cuda_error */
  SWZ_ETIMEOUT = -5,       /* a bounded device wait expired (swz_check_status)*/
  SWZ_EUNSUPPORTED = -6,   /* valid arguments, configuration not provided     */
  SWZ_ESCRATCH = -7        /* launch needs more than the library's built-in
                              scratch area (swz_gemm_streamk_noalloc)        */
};

/* ---- tile orders ([TBS] mode ids 0..4; 5 added for [CPS] serpentine) ----- */
enum swz_order {
  SWZ_ROW = 0,        /* m = id / gn, n = id % gn                              */
  SWZ_COL = 1,        /* m = id % gm, n = id / gm                              */
  SWZ_PANEL = 2,      /* grouped 2D panel, G rows per band (= [CPS] group-major)*/
  SWZ_MORTON = 3,     /* bit 2i of id -> bit i of m, bit 2i+1 -> bit i of n    */
  SWZ_XOR = 4,        /* m = ((id % gn) ^ (id / gn)) % gm, n = (id / gn) % gn  */
  SWZ_SERPENTINE = 5  /* strips of S columns, rows walked down / up alternately*/
};

/* operand types: fp16, bf16, or fp32 multiplied as TF32 (the first page's
 * --dtype fp32 runs the same kernel with TF32 tensor cores) */
enum swz_dtype { SWZ_F16 = 0, SWZ_BF16 = 1, SWZ_TF32 = 2 };

/* storage of B: K x N row-major (the pages' B) or N x K row-major (B
 * transposed, K contiguous) */
enum swz_b_layout { SWZ_B_KN = 0, SWZ_B_NK = 1 };

/* shared-memory tile layouts of the transpose ([SBC] "Matrix Transpose") */
enum swz_smem_layout {
  SWZ_SMEM_NAIVE = 0,   /* tile[32][32], element (r,c) at r*32 + c            */
  SWZ_SMEM_PADDED = 1,  /* tile[32][33], element (r,c) at r*33 + c            */
  SWZ_SMEM_XOR = 2      /* tile[32][32], element (r,c) at r*32 + (c ^ r)      */
};

/*
 * swz_tile_map -- [TBS] tile-order functions, [CPS] serpentine.
 * For every program id p in [0, grid_m*grid_n) writes d_m[p], d_n[p]: the
 * output tile (row, column) that `order` maps p to, computed on the device by
 * the same function the GEMM's scheduler calls.  `group` is G for SWZ_PANEL
 * and S for SWZ_SERPENTINE (>= 1), ignored otherwise.  d_m, d_n: device int32
 * arrays of grid_m*grid_n entries.  Morton/XOR maps are written even when not
 * bijective (the map is well defined; only the GEMM refuses them).
 * Errors: SWZ_EINVAL (grid <= 0, grid_m*grid_n > 2^31-1, group < 1 where
 * used, null arrays, unknown order), SWZ_EARCH, SWZ_ECUDA.
 */
int swz_tile_map(int order, int grid_m, int grid_n, int group,
                 int32_t* d_m, int32_t* d_n, void* stream);

/* Host-side check: 1 if `order` visits each of the grid_m x grid_n tiles
 * exactly once, 0 if not, SWZ_EINVAL on bad arguments. */
int swz_is_bijective(int order, int grid_m, int grid_n, int group);

/*
 * swz_gemm -- [TBS] benchmark GEMM: C = A * B with FP32 accumulation.
 * A: M x K, B: K x N, both row-major fp16 on the device; C: M x N row-major
 * FP32 (written, never read).  Output tiles are 128 x 256 (128 x 128 when
 * N <= 128), visited in `order` (group = G or S as in swz_tile_map).
 * persistent = 0: one CTA per output tile, tile = order(blockIdx.x) ([TBS]
 * non-persistent launch); persistent = 1: min(tiles, resident CTAs) CTAs,
 * CTA b takes tile ids b, b + P, b + 2P, ... ([TBS] persistent loop, [CPS]
 * work_idx striding).  Ragged M, N, K are handled (TMA zero-fill on loads,
 * clipped stores).  K = 0 writes zeros; M = 0 or N = 0 is a no-op.
 * Summation order: a tile's K blocks are accumulated in ascending order,
 * except that in a persistent launch the whole tiles of every other wave
 * (tile id / P odd, P = programs, or clusters with cta_pair) take them in
 * descending order, so that each wave starts on the operand slices the
 * previous wave read last (fewer DRAM reads).  The order depends on the
 * tile id and P only: results are deterministic, equal for the static and
 * dynamic schedulers and the die split, and between launches with another
 * P agree up to FP32 rounding order.
 * Launches allow programmatic dependent launch: the kernel may start while
 * the previous kernel of `stream` finishes, and touches no global memory
 * before that kernel has completed.
 * Requirements: A, B 16-byte aligned; C 16-byte aligned; rows of A (and of
 * B in either layout) a multiple of 16 bytes (K % 8 == 0 for fp16/bf16,
 * K % 4 == 0 for TF32; N % 8 == 0 for B as K x N); N % 4 == 0; M, N, K <
 * 2^31.  Errors: SWZ_EINVAL, SWZ_ENOTBIJECTIVE (Morton
 * or XOR on a grid they do not permute), SWZ_EARCH, SWZ_ECUDA.
 */
int swz_gemm(const void* A, const void* B, float* C, int M, int N, int K,
             int order, int group, int persistent, void* stream);

/* Options of swz_gemm_ex (zero-initialise, then set what you need). */
typedef struct swz_gemm_opts {
  int dtype;         /* SWZ_F16 (default), SWZ_BF16 or SWZ_TF32 (fp32 A and B,
                        multiplied as TF32; needs b_layout = SWZ_B_NK)        */
  int tile_n;        /* 128 or 256; 0 = automatic as in swz_gemm             */
  int cta_pair;      /* 1: 2-CTA clusters, tcgen05 cta_group::2, cluster tile
                        256 x tile_n (tile_n 256, the default, or 128; each
                        CTA owns 128 x tile_n of C) -- [CPS] Example 2;
                        0: single CTA                                        */
  int num_programs;  /* persistent only: CTAs to launch (a multiple of 2 with
                        cta_pair); 0 = resident capacity;
                        capped at the tile count (scheduler units) except
                        with stream_k, where a launch with fewer units than
                        programs splits each unit's K among programs      */
  int32_t* d_trace;  /* optional device array, 2 int32 per CTA tile, indexed
                        (cta_m * tiles_n + cta_n): {program (blockIdx.x),
                        iteration of that program's tile loop}               */
  uint32_t debug_flags; /* SWZ_DEBUG_*; 0 in normal use                      */
  uint32_t timeout_ms;  /* bound of every device wait; 0 = 2000 ms           */
  int stream_k;      /* persistent only: 1 = share the last, partial wave of
                        tiles among all programs by splitting those tiles'
                        K iterations into equal contiguous ranges (Stream-K;
                        with fewer tiles than programs every tile is split);
                        needs d_workspace of swz_gemm_workspace_size bytes   */
  void* d_workspace; /* device scratch for stream_k: partial accumulators and
                        per-piece flags.  Zero-fill it once before its first
                        use; the library keeps it consistent afterwards
                        (in graph replays too: a captured call clears the
                        flags before its launch).  Launches sharing a
                        workspace must not overlap.                          */
  uint64_t workspace_bytes; /* size of d_workspace                           */
  int b_layout;      /* SWZ_B_KN (default): B is K x N row-major; SWZ_B_NK: B
                        is stored transposed, N x K row-major (K contiguous)  */
  int smem_swizzle;  /* span in bytes of the TMA / tensor-core shared-memory
                        swizzle of the operand stages ([SBC] "Hopper TMA 的
                        swizzling": the 16-byte chunk index of an address is
                        XORed with the bits just above the span): 128
                        (default when 0), 64 or 32.  Same results and stage
                        bytes in every mode; with 64 and 32 a 128-byte row of
                        a stage is split into 2 or 4 column groups of the
                        span's width.  The C staging keeps the 128-byte span. */
  int dynamic;       /* persistent only, not with stream_k, span 128 only:
                        tiles are claimed at run time instead of dealt out by
                        work_idx striding.  1: program c takes work index c
                        first, then P + the value of an atomic counter it
                        increments (P = programs, or clusters with cta_pair),
                        until the indices run out.  Each index goes through
                        the tile order as usual.  The counter lives at the
                        start of d_workspace (256-byte aligned, at least
                        swz_gemm_workspace_size bytes = 256) and is cleared on
                        `stream` before the launch; launches sharing a
                        workspace must not overlap.                          */
  int die_split;     /* persistent only, not with dynamic: 1 = split the work
                        between the two dies of the package.  The clusters on
                        die 0 take the first U0 scheduler units of the tile
                        order and the clusters on die 1 the rest (U0 = the
                        units times die 0's share of the clusters, rounded),
                        each die striding (and with stream_k splitting its own
                        tail) over its own clusters, so that most operand
                        lines are read by the SMs of one die.  Needs
                        swz_calibrate on the device first (SWZ_EUNSUPPORTED
                        otherwise).  Applies to launches at the resident
                        capacity (num_programs 0); other launches, and a
                        device whose SMs all sit on one die, run the plain
                        schedule.  The die of each cluster only decides which
                        tiles it takes (see swz_gemm_die_plan): whole tiles
                        are those of the plain schedule bit for bit; with
                        stream_k each die splits its own tail, so other tiles
                        are split at other K blocks than in the plain
                        schedule (the same result up to FP32 summation order,
                        deterministic from run to run).  0: off              */
} swz_gemm_opts;

/* debug_flags: withhold the first operand load so that the consumer's
 * bounded wait expires; the kernel then records SWZ_ETIMEOUT for
 * swz_check_status and exits cleanly (tests of the timeout path only). */
#define SWZ_DEBUG_SKIP_FIRST_LOAD 1u

/* swz_gemm with explicit tile shape, dtype, 2-CTA mode, program count, trace,
 * wait bound and Stream-K tail.  opts may be NULL (= swz_gemm).  Extra
 * errors: SWZ_EUNSUPPORTED for tile_n not in {0,128,256}, or stream_k
 * with more programs than can be resident at once (its pieces wait on one
 * another); SWZ_EINVAL for stream_k without persistent or with a missing,
 * misaligned (256 B) or too small workspace, and for smem_swizzle not in
 * {0, 32, 64, 128}; for dynamic the same workspace rules, SWZ_EINVAL for a
 * value other than 0 or 1, without persistent or with stream_k,
 * SWZ_EUNSUPPORTED with a span other than 128; for die_split SWZ_EINVAL for
 * a value other than 0 or 1, without persistent or with dynamic,
 * SWZ_EUNSUPPORTED on a device swz_calibrate has not measured.
 * In Stream-K mode the trace records, for a split tile, the program that
 * wrote it. */
int swz_gemm_ex(const void* A, const void* B, float* C, int M, int N, int K,
                int order, int group, int persistent,
                const swz_gemm_opts* opts, void* stream);

/*
 * swz_gemm_host -- the [TBS] GEMM from host memory: C = A * B with A, B read
 * from host buffers and C written to a host buffer, the copies overlapped
 * with the computation.  B (K x N) is copied to d_B first; A and C are cut
 * into `slabs` row slabs (0 = 4; at most 64; slab heights are multiples of
 * 256 rows): slab i of A is copied in on an input stream, multiplied on
 * `stream` by swz_gemm_ex (persistent = 1, opts as given, order/group within
 * the slab), and slab i of C copied out on an output stream while later
 * slabs proceed.  The call is asynchronous like the others: when `stream`
 * reaches the point after the call, C is in h_C.
 * h_A (M x K), h_B (K x N): host, fp16/bf16 per opts->dtype; h_C (M x N,
 * fp32): host.  Pinned (page-locked) host buffers are needed for the copies
 * to overlap.  d_A, d_B, d_C: caller-owned device buffers of the full sizes,
 * 16-byte aligned; their contents are overwritten.  The library keeps two
 * streams and some events per device for this call (no device memory); calls
 * are serialised while they enqueue.  Host-side argument and configuration
 * checks (including Morton/XOR bijectivity on every slab grid) happen before
 * anything is enqueued; a CUDA failure part-way returns SWZ_ECUDA with the
 * earlier copies already enqueued.  Errors: as swz_gemm_ex.
 */
int swz_gemm_host(const void* h_A, const void* h_B, float* h_C, int M, int N, int K,
                  int order, int group, const swz_gemm_opts* opts, void* d_A, void* d_B,
                  float* d_C, int slabs, void* stream);

/* Bytes of d_workspace a launch with these arguments needs (0 when
 * stream_k is off, the launch is not persistent or the tiles divide evenly
 * among the programs).  Needs the device when persistent and num_programs is
 * 0 (resident capacity). */
int swz_gemm_workspace_size(int M, int N, int K, int persistent,
                            const swz_gemm_opts* opts, uint64_t* h_bytes);

/*
 * swz_calibrate -- finds, on the current device, which die of the package
 * each SM sits on and where each persistent GEMM kernel shape places its
 * CTAs, for the die_split schedule.  No source page has a counterpart: it
 * is a GB300 property (two dies, each with half of the L2; a line one die's
 * SM has read is a slower L2 hit for the other die's SMs).
 *
 * The die of an SM is found by timing: one CTA reads a buffer into its half
 * of the L2, then one CTA per SM times a chain of dependent loads through
 * its own slice; the SMs of the other die see the cross-die latency.  The
 * placement is recorded by launching each kernel shape once at its resident
 * capacity (the hardware places persistent CTAs the same way every time).
 * The call is synchronous: it allocates and frees temporary device buffers
 * (about 16 KB per SM), launches the probe kernels and waits for them.
 * Results are kept per device for the life of the process; calling again
 * repeats the measurement.
 *   h_die_of_sm  host, max_sms ints (may be NULL with max_sms 0): the die
 *                (0 or 1) of SM id s at [s]; all 0 on a single die
 *   h_num_sms    host, optional: the device's SM count
 * Errors: SWZ_EINVAL, SWZ_EARCH, SWZ_ECUDA, SWZ_EUNSUPPORTED (not every SM
 * could be measured, e.g. while other work occupies the device).
 */
int swz_calibrate(int* h_die_of_sm, int max_sms, int* h_num_sms);

/* The die split a persistent launch with these arguments would use
 * (opts->die_split need not be set): for each cluster g (CTAs g*c .. g*c +
 * c - 1, c = 2 with cta_pair) h_cluster_info[g] = die << 15 | rank of the
 * cluster among its die's clusters, h_P0 = die 0's clusters, h_U0 = the
 * scheduler units die 0 takes, h_clusters = the launch's clusters.  When the
 * launch gets no split, every cluster reads as die 0 with rank g, P0 = the
 * clusters and U0 = the units.  Errors: SWZ_EINVAL, SWZ_EUNSUPPORTED (device
 * not calibrated), as swz_gemm_plan otherwise. */
int swz_gemm_die_plan(int M, int N, int K, const swz_gemm_opts* opts,
                      int32_t* h_cluster_info, int max_clusters, int* h_clusters,
                      int* h_P0, int* h_U0);

/* Grid and launch the GEMM would use, without launching: tiles_m, tiles_n
 * (CTA tiles), sched_m, sched_n (scheduler grid: cluster tiles in 2-CTA mode)
 * and programs (CTAs launched).  Any out pointer may be NULL. */
int swz_gemm_plan(int M, int N, int K, int persistent,
                  const swz_gemm_opts* opts, int* tiles_m, int* tiles_n,
                  int* sched_m, int* sched_n, int* programs);

/*
 * swz_gemm_mma_sync -- [TBS] GEMM C = A * B (as swz_gemm: A M x K, B K x N
 * row-major fp16/bf16 per `dtype`, C M x N fp32) on the warp-level tensor-core
 * path: cp.async into shared memory, ldmatrix fragments, mma.sync m16n8k16,
 * 128 x 128 x 64 CTA tiles, one CTA per tile in `order` (group as in
 * swz_gemm).  The operand tiles' shared-memory layout is chosen by
 * (vec, per_phase, max_phase, pad): element (r, c) of a tile with rows of W
 * elements sits at r*(W + pad) + ((c/vec) ^ ((r/per_phase) % max_phase))*vec
 * + c % vec -- [SBC] "Triton - Shared Layout swizzling" plus "Padding";
 * (8,1,1,0) is the plain layout, (8,1,8,0) the 128-byte swizzle
 * (Swizzle<3,3,3>, [SBC] "swizzle in CUTLASS"), (8,2,4,0) a 64-byte-style
 * swizzle, (8,1,1,8) 16-byte padding.  Results are identical for every
 * layout; ldmatrix bank conflicts ([SBC] "MMA Bank Conflict") are not.
 * Requirements: vec, per_phase, max_phase powers of two, vec a multiple of
 * 8, max_phase * vec <= 64, pad in {0, 8, ..., 64}; K % 8 == 0, N % 8 == 0;
 * A, B 16-byte and C 8-byte aligned.  K = 0 writes zeros.  Errors:
 * SWZ_EINVAL, SWZ_ENOTBIJECTIVE, SWZ_EARCH, SWZ_ECUDA.
 */
int swz_gemm_mma_sync(const void* A, const void* B, float* C, int M, int N, int K,
                      int dtype, int vec, int per_phase, int max_phase, int pad,
                      int order, int group, void* stream);

/*
 * swz_transpose -- [SBC] "Matrix Transpose": out[j][i] = in[i][j] for an
 * M x N matrix of 32-bit words (out is N x M, row-major), staged through a
 * 32 x 32 shared-memory tile in `layout` (swz_smem_layout).  The result is
 * bit-identical for all layouts; they differ in shared-memory bank conflicts
 * (naive: 31 per warp store; padded and XOR: none).  Any M, N >= 0 (ragged
 * edges clipped; 0 = no-op), M, N <= 2^31-1 with M*N < 2^62 and M/32 < 65536
 * tiles along M.  in, out: device, 4-byte aligned, must not overlap.
 * Errors: SWZ_EINVAL, SWZ_EARCH, SWZ_ECUDA.
 */
int swz_transpose(const uint32_t* in, uint32_t* out, int M, int N, int layout,
                  void* stream);

/*
 * swz_l2_model -- [TBS] benchmark, offline L2 model (host only, no GPU).
 * Replays the tile order's operand-tile trace through a byte-budget LRU
 * cache: the L2 holds whole tiles (A: tile_m x tile_k, B: tile_k x tile_n
 * elements of elem_bytes), a hit refreshes a tile, a miss inserts it and then
 * evicts least-recently-used tiles while more than l2_bytes are held and more
 * than one tile is held.  Program ids run in waves of `concurrency` CTA
 * tiles; within a wave, for every K step, each tile touches A(m, k) then
 * B(k, n).  cluster_m > 1 runs the order on cluster tiles of
 * cluster_m x 1 CTA tiles (the [CPS] Example 2 split), each cluster tile
 * contributing its CTA tiles in rank order.  Writes the hit and miss counts;
 * hit rate = hits / (hits + misses).  Errors: SWZ_EINVAL.
 */
int swz_l2_model(int order, int group, int M, int N, int K, int tile_m, int tile_n,
                 int tile_k, int elem_bytes, int64_t l2_bytes, int concurrency,
                 int cluster_m, int64_t* h_hits, int64_t* h_misses);

/* swz_l2_model plus the bytes the misses bring in (each miss of an A tile
 * counts tile_m * tile_k * elem_bytes, of a B tile tile_k * tile_n *
 * elem_bytes): the model's prediction of the operand bytes read from DRAM.
 * l2_partitions = 1 is the [TBS] model.  l2_partitions = p > 1 models an L2
 * split into p halves, one per die (GB300: 2), where every operand line is
 * read by SMs of every die and each half keeps its own copy: each half
 * replays the whole trace with l2_bytes / p of capacity, and the counts are
 * those of one half.  This is a reading of the hardware, not the page's
 * model.  k_alternate = 1 replays the K order of swz_gemm's persistent
 * launches instead of the page's: the tiles of odd waves take the K steps
 * from the last to the first (0: every wave ascending, the page's model).
 * Errors: SWZ_EINVAL (as swz_l2_model, l2_partitions < 1, k_alternate not 0
 * or 1, or h_miss_bytes NULL). */
int swz_l2_model_bytes(int order, int group, int M, int N, int K, int tile_m, int tile_n,
                       int tile_k, int elem_bytes, int64_t l2_bytes, int l2_partitions,
                       int k_alternate, int concurrency, int cluster_m, int64_t* h_hits,
                       int64_t* h_misses, int64_t* h_miss_bytes);

/*
 * swz_gemm_streamk_noalloc -- Stream-K GEMM for callers that cannot allocate
 * device memory.  No source page has a counterpart; this is a library
 * convenience.
 *
 * Who needs it: callers that are handed only their input and output buffers
 * and have no way to get device scratch -- plugin hosts that own every
 * allocation, services running under a fixed memory budget whose allocator
 * belongs to someone else, and loops that must not call cudaMalloc because
 * it synchronises the device.  swz_gemm_ex with stream_k needs a
 * caller-provided workspace; this entry point instead uses a scratch area
 * built into the library: a statically sized device array of
 * SWZ_NOALLOC_SCRATCH_BYTES (40 MiB) that every GPU which loads the library
 * holds until the process exits.
 *
 * Computes exactly what swz_gemm_ex computes with persistent = 1, stream_k =
 * 1 and the same opts (dtype, tile_n, cta_pair, num_programs, d_trace,
 * timeout_ms; opts->stream_k, d_workspace and workspace_bytes are ignored;
 * opts may be NULL).  A, B, C as in swz_gemm.
 *
 * Set-up: the first call on each device looks up the device address of the
 * scratch area (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept for the life of
 * the process and does not survive cudaDeviceReset (or anything else that
 * destroys the device's primary context): do not call this entry point on a
 * device after resetting it.  The call allocates and frees nothing.  It clears the part of the scratch area that must start at zero
 * (the per-piece flags) on `stream` before the launch.
 *
 * All calls on a device share the one scratch area, which keeps the last
 * call's contents: calls whose work overlaps on the GPU (different streams,
 * or host threads racing on one device) race on it and must be serialised
 * by the caller.
 *
 * Errors: as swz_gemm_ex, plus SWZ_ESCRATCH when the launch needs more than
 * SWZ_NOALLOC_SCRATCH_BYTES of scratch (see swz_gemm_workspace_size).
 */
#define SWZ_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)
int swz_gemm_streamk_noalloc(const void* A, const void* B, float* C, int M, int N, int K,
                             int order, int group, const swz_gemm_opts* opts,
                             void* stream);

/*
 * swz_tc_rate -- measures the dense tensor-core rate of this library's
 * tcgen05 MMA code, for the roofline denominator.  No source page has a
 * counterpart: the pages quote peak figures; this measures FLOP per SM clock.
 *
 * Launches num_ctas CTAs (0 = one per SM; at most the SM count, one CTA per
 * SM).  Each copies A and B into shared memory (128-byte swizzle, as the
 * GEMM stages its operands) and issues n_mma tcgen05.mma instructions of
 * shape 128 x n x k (k = 16 for SWZ_F16 / SWZ_BF16, 8 for SWZ_TF32), the i-th
 * on k-slice i % 4 of the operands, all accumulating into one fp32 TMEM
 * accumulator (the first overwrites it).  One instruction is 2 * 128 * n * k
 * FLOP; there is no global-memory traffic while it runs.
 *   dtype   SWZ_F16, SWZ_BF16 or SWZ_TF32 (A and B of that type).
 *   n       MMA N: 64, 128 or 256.
 *   A       device, 128 rows x 128 bytes, row-major (64 fp16/bf16 or 32 fp32
 *           per row): the 128 x 4k operand, K-major.
 *   B       device, n rows x 128 bytes, row-major: B stored N x K.
 *   n_mma   instructions per CTA, 1 .. 2^24.
 *   d_times device, 4 * ctas uint64, written per CTA c at 4c: SM cycles from
 *           the first issue to completion, globaltimer ns over the same span,
 *           the SM id, and 0 (completed) or 1 (the bounded wait for
 *           completion expired; the other fields are then not a rate).
 *   d_D     device fp32 128 x n, or NULL: CTA 0's accumulator at the end;
 *           with n_mma % 4 == 0 it is (n_mma / 4) * A * B^T (A, B as read
 *           in the dtype; TF32 keeps 10 fraction bits of each fp32 operand).
 * FLOP / clock / SM = n_mma * 2 * 128 * n * k / cycles.  Pointers 16-byte
 * (A, B), 8-byte (d_times) and 4-byte (d_D) aligned.  Errors: SWZ_EINVAL,
 * SWZ_EARCH, SWZ_ECUDA.
 */
int swz_tc_rate(int dtype, int n, const void* A, const void* B, int n_mma, int num_ctas,
                uint64_t* d_times, float* d_D, void* stream);

/*
 * swz_tc_rate_ex -- swz_tc_rate (= cta_pair 0, mmas_per_stage 0) with two
 * more shapes of the issue loop, to measure what the GEMM's single issuing
 * thread can sustain:
 *   cta_pair        1: 2-CTA clusters, tcgen05 cta_group::2 MMAs of 256 x n x
 *                   k issued by the even CTA of each pair; CTA 2i+r holds A
 *                   (both CTAs the same 128 rows) and B rows r*n/2 .. +n/2-1.
 *                   n 128 or 256; num_ctas even (0 = the SM count rounded
 *                   down to even).
 *   mmas_per_stage  0: n_mma MMAs back to back.  4, 8 or 16: the loop is cut
 *                   into stages as in the GEMM -- per stage a non-blocking
 *                   test of a barrier whose phase is already complete (it
 *                   never waits), the tensor fence, that many MMAs and a
 *                   commit -- unrolled by 8; n_mma % mmas_per_stage == 0.
 * d_times holds one record per issuing CTA (num_ctas / 2 with cta_pair), in
 * the format of swz_tc_rate; d_D is CTA 0's accumulator (rows 0..127 of a
 * pair's 256) with the same identity.  FLOP / clock / SM = n_mma * 2 * 128 *
 * n * k / cycles in both modes (a pair's MMA is two SMs' work).  Errors: as
 * swz_tc_rate; SWZ_EINVAL for cta_pair or mmas_per_stage out of range;
 * SWZ_EUNSUPPORTED for SWZ_TF32 with a pair or stages.
 */
int swz_tc_rate_ex(int dtype, int n, int cta_pair, int mmas_per_stage, const void* A,
                   const void* B, int n_mma, int num_ctas, uint64_t* d_times, float* d_D,
                   void* stream);

/* Synchronises `stream`, then returns and clears the current device's
 * status word: SWZ_OK, or SWZ_ETIMEOUT if a kernel's bounded wait expired
 * since the last check. */
int swz_check_status(void* stream);

/* Static description of a status code (never NULL). */
const char* swz_strerror(int status);

/* cudaError_t of the last failing CUDA call in this thread (0 if none). */
int swz_last_cuda_error(void);

/* Properties of the current device the scheduler uses: SM count, L2 bytes,
 * compute capability.  Out pointers may be NULL. */
int swz_device_info(int* num_sms, int* l2_bytes, int* cc_major, int* cc_minor);

#ifdef __cplusplus
}
#endif
#endif /* SWZ_H_ */
