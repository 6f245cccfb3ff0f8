// Kernel parameter blocks (passed by value as __grid_constant__) and the
// host-side launch entry points of each kernel translation unit.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bwg {

constexpr int kThreads = 192;        // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kThreads2C = 384;      // two-consumer pair kernel: 12 warps
// Registers per thread of the two-consumer kernel: at launch (one CTA per SM,
// 65,536 / 384 rounded down to a multiple of 8), and the split after set-up
// between warpgroup 0 (TMA, MMA) and the two epilogue warpgroups.
constexpr uint32_t kRegsLaunch2C = 168;
constexpr uint32_t kRegsControl2C = 56;
constexpr uint32_t kRegsEpilogue2C = 224;
static_assert(kRegsControl2C * 128 + kRegsEpilogue2C * 256 <= kRegsLaunch2C * kThreads2C,
              "the register split must fit in the launch allocation");
static_assert(kRegsLaunch2C * kThreads2C <= 65536, "one CTA per SM");
constexpr int kBK = 64;              // K per stage: one 128-byte swizzle row of 16-bit data
constexpr int kTileN = 256;          // output columns per tile (MMA N)
constexpr int kRowsPerCta = 128;     // accumulator rows per CTA (TMEM lanes)
constexpr int kEpiBufBytes = 4096;   // one 32-row x 128-byte staging box
constexpr int kEpiBytes = 4 * 2 * kEpiBufBytes;  // 4 epilogue warps, double-buffered
constexpr uint32_t kTmemCols = 512;  // two 256-column FP32 accumulators
constexpr int kMaxGroupsPerLaunch = 64;
constexpr int kSmallMMaxM = 128;     // swapped kernel handles up to 128 rows of A
constexpr int kMaxSplit = 8;         // largest cluster of the small-M split (portable size)

// Output element type codes (same values as the C ABI).
constexpr int kOutBF16 = 0;
constexpr int kOutF32 = 1;
constexpr int kOutF16 = 2;

// Device error word layout (written once per fault with atomicCAS from 0):
//   [56,64) kind (1 = barrier wait timed out, 2 = invalid group offsets)
//   [48,56) role (0 TMA producer, 1 MMA issuer, 2 epilogue)
//   [40,48) barrier (0 full, 1 empty, 2 accumulator full, 3 accumulator empty)
//   [16,40) block index      [8,16) stage      [0,8) phase parity
constexpr unsigned long long kFaultTimeout = 1;
constexpr unsigned long long kFaultBadOffsets = 2;

struct GemmParams {
  CUtensorMap map_a;  // A [rows, K] bf16/fp16, box {64 (K), 128 (rows)}, 128B swizzle
  CUtensorMap map_b;  // B [K, N], box {64 (N), 64 (K)}; or B [N, K] (b_kmajor), box {64 (K), 64 (N)};
                      // 128B swizzle (dense only)
  CUtensorMap map_d;  // D [rows, N], box {64 or 32 (N), 32 (rows)}, 128B swizzle
  // B, one load for a pair CTA's 128 columns of a stage (b_one_box): [K, N]
  // as a 3-D view {64 (N in a chunk), K, N/64 chunks} with box {64, 64, 2};
  // [N, K] (b_kmajor) as 2-D with box {64 (K), 128 (N)}.  Either lands exactly
  // as the two 64-column boxes of map_b would.
  CUtensorMap map_b1;
  int b_one_box;      // 1: map_b1 is valid and the pair kernels use it (dense only)
  unsigned long long* err;
  void* d_ptr;               // D base, for masked row stores at ragged group ends
  const int* group_offsets;  // grouped only: device int32 [G+1]
  unsigned long long timeout_ns;
  int M, N, K, ldd;          // M = rows of A and D (total rows for grouped)
  int num_m_tiles, num_n_tiles, num_k_blocks;
  int group_m;               // raster: tile rows per group of the grouped order
  int stages;
  int out_dtype;
  uint32_t idesc;
  uint32_t tx_extra;         // test hook: extra bytes expected per stage (0 normally)
  int G, g_begin, G_total;   // grouped only: groups in this launch, first group, all groups
  int no_tail_split;         // 1: never split last-wave tiles (tests and measurements)
  int direct_store;          // 1: epilogue stores rows from registers (no staging, one more stage)
  int swap_ends;             // grouped: 1 = compute group ends of <= 128 rows with swapped operands
  uint32_t idesc_swap;       // grouped: descriptor of the swapped MMA (A MN-major, B K-major)
  int swiglu_up;             // SwiGLU kernels: first column of the up block in B (= N of H)
  int b_kmajor;              // 1: B is stored [N, K] (K-major operand), 0: [K, N]
  int workers;               // dynamic scheduling: CTA pairs that run at once (last-wave cut)
  // Stream-K last wave (dense two-consumer kernel, static schedule): the last
  // sk_tiles tiles of the raster order are shared out by k-blocks over all
  // pairs; each pair first works through its k-block range (at most sk_segs
  // segments), then its whole tiles.
  int sk_tiles;              // 0: no stream-K
  int sk_segs;
  int ws_slots;              // partial slots per stream-K tile (most pairs sharing one)
  float* ws;                 // partials [sk_tiles][ws_slots][16 warp slices][32 rows][256] FP32
  int* ws_counters;          // arrivals [sk_tiles][16 warp slices], zero between calls
  // Optional unit trace (nullptr: off): per CTA, kTraceUnits records of
  // kTraceWords words (global timer, ns).
  unsigned long long* trace;
};

constexpr int kTraceUnits = 64;
constexpr int kTraceWords = 5;  // unit, producer start, epilogue end, accumulator seen, released

struct GroupedParams {
  GemmParams base;
  CUtensorMap map_b[kMaxGroupsPerLaunch];
};

struct SmallMParams {
  // One ring stage of B^T (the MMA's A operand, 128 channels x 64 K):
  //  - row-major B [K, N], bt_boxes == 1: a 3-D view {64 channels, K, N/64
  //    channel groups} (strides ldb*2 and 128 bytes), box {64, 64, 2}: both
  //    64-channel halves of the stage in one load;
  //  - row-major B, bt_boxes == 2 (N not a multiple of 64): 2-D {N, K}, box
  //    {64, 64}, one load per half;
  //  - B stored [N, K] (b_kmajor): 2-D {K, N}, box {64 (K), 128 (rows)}.
  CUtensorMap map_bt;
  CUtensorMap map_at;  // A [M, K] as the MMA's K-major B: box {64 (K), m_pad (rows)}
  // Two consecutive ring stages in one load each (pair_loads): B^T as a 4-D
  // view {64, 64, N/64, K/64} with box {64, 64, 2, 2} (row-major B) or a 3-D
  // view {64 (K), N, K/64} with box {64, 128, 2} (B [N, K]); A as a 3-D view
  // {64 (K), M, K/64} with box {64, m_pad, 2}.  Each lands exactly as two
  // single-stage loads would.
  CUtensorMap map_bt2;
  CUtensorMap map_at2;
  CUtensorMap map_d;   // D [M, N], box {min(64, tile_n) (N), m_pad (rows)}, no swizzle
  CUtensorMap map_d2;  // D [M, N], box {tile_n - 64 (N), m_pad}, when tile_n > 64
  unsigned long long* err;
  unsigned long long timeout_ns;
  int M, N, K, m_pad;
  int tile_n;          // output columns per tile (<= 128; the MMA always spans 128)
  int num_tiles, num_k_blocks, stages, out_dtype;
  uint32_t idesc;
  uint32_t tx_extra;
  int streamk;       // 1: (tile, k-block) iterations shared evenly over the grid
  int ws_slots;      // partial-accumulator slots per tile (most CTAs sharing a tile)
  float* ws;         // stream-K partials: [num_tiles][ws_slots][m_pad][128] FP32
  int* ws_counters;  // stream-K arrival counters, one per tile, zero between calls
  // Cluster split of K (split > 1): the grid is num_tiles clusters of `split`
  // CTAs; CTA r of cluster t computes k-blocks [r*kb/split, (r+1)*kb/split) of
  // tile t, and the cluster sums its partials through distributed shared
  // memory, each CTA finishing ceil(M/split) rows of D, which it stores itself.
  int split;
  int b_kmajor;         // 1: B is stored [N, K]
  int staging_in_ring;  // 1: one tile per CTA, the output staging tile sits in the idle ring
  int bt_boxes;         // loads per single stage of B^T (1 or 2), see map_bt
  int pair_loads;       // 1: fill stages s, s+1 (s even) with map_bt2 / map_at2 where two
                        // k-blocks of the segment remain
  int l2hint;           // L2 policies: bit 1 loads B^T evict-first (the default), bit 0
                        // loads A evict-last; evict-normal where a bit is clear
  void* d;            // D (split mode stores its rows directly)
  long long ldd;      // D's leading dimension, elements
  // Optional trace (nullptr: off): per CTA eight global-timer stamps (ns),
  // documented with bwg_debug_set_trace.
  unsigned long long* trace;
};

// Host launchers (one per kernel instantiation).  They only enqueue.
cudaError_t launch_gemm_1cta(const GemmParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_gemm_2cta(const GemmParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_gemm_2cta_mc(const GemmParams& p, int grid, size_t smem, cudaStream_t s);
// dynamic: cluster-launch-control scheduling (grid = one pair per unit)
cudaError_t launch_gemm_2cta_2c(const GemmParams& p, int grid, size_t smem, cudaStream_t s,
                                bool dynamic = false);
int max_active_clusters_gemm_2c(size_t smem);
// Grouped launchers; swiglu = the fused SwiGLU epilogue over a [gate | up] B.
cudaError_t launch_grouped_2c(const GroupedParams& p, int grid, size_t smem, cudaStream_t s,
                              bool swiglu = false, bool dynamic = false);
int max_active_clusters_grouped_2c(size_t smem);
cudaError_t launch_grouped_2cta(const GroupedParams& p, int grid, size_t smem, cudaStream_t s,
                                bool swiglu = false);
cudaError_t launch_small_m(const SmallMParams& p, int grid, size_t smem, cudaStream_t s);
// Co-resident clusters of `cluster` small-M CTAs with `smem` bytes each (0 on error).
int max_active_clusters_small_m(int cluster, size_t smem);
cudaError_t launch_zero_fill(void* d, int rows, int cols, int ld, int elt_bytes, cudaStream_t s);

// Probe kernels (test hooks, probes.cu).
cudaError_t launch_probe_cluster_pair(const float* in, float* sum_out, int* peer_out, int n,
                                      cudaStream_t s);
cudaError_t launch_probe_tma_swizzle(const CUtensorMap& map, void* out, unsigned long long* err,
                                     unsigned long long timeout_ns, cudaStream_t s);
cudaError_t launch_probe_grouped_tables(const int* offsets, int g0, int G, int G_total, int M,
                                        int num_n_tiles, int tile_m, int* out, cudaStream_t s);
cudaError_t launch_probe_mma(const CUtensorMap& map_a, const CUtensorMap& map_b, float* d, int k_steps,
                             uint32_t idesc, unsigned long long* err, unsigned long long timeout_ns,
                             cudaStream_t s);

// Occupancy helpers: co-resident clusters (or CTAs) for a given launch shape.
int max_active_clusters_gemm(int cluster, bool grouped, size_t smem);
int max_active_ctas_small_m(size_t smem);

}  // namespace bwg
