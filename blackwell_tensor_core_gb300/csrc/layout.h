// Bit layouts shared by the host planner/tests and the kernels:
//  - the tcgen05.mma instruction descriptor for kind::f16,
//  - the tcgen05 shared-memory matrix descriptor,
//  - the 128-byte swizzle that TMA applies to a tile in shared memory.
//
// Field positions follow the public PTX ISA (tcgen05 "Instruction descriptor"
// and "Shared memory descriptor" tables).  The MegaMoE page ("MegaMoE …
// 融合算子解读", section 04, dynamic N) prints one of these fields itself: the
// N extent enters the instruction descriptor as (N >> 3) << 17.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define BWG_HD __host__ __device__ __forceinline__
#else
#define BWG_HD inline
#endif

namespace bwg {

// Operand formats of kind::f16 (A and B must share one of these).
constexpr uint32_t kFmtF16 = 0;
constexpr uint32_t kFmtBF16 = 1;

// Instruction descriptor, kind::f16, FP32 accumulator:
//   [4,6)  D format (1 = F32)       [7,10) A format     [10,13) B format
//   15     A is MN-major            16     B is MN-major
//   [17,23) N >> 3                  [24,29) M >> 4
BWG_HD uint32_t make_idesc_f16(uint32_t ab_fmt, bool a_mn_major, bool b_mn_major, uint32_t m,
                               uint32_t n) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Swizzle modes of the shared-memory descriptor (bits 61..63).
constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// Shared-memory matrix descriptor:
//   [0,14)  start address >> 4      [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4 [46,48) version (1 for tcgen05)
//   [49,52) base offset (0: tiles are 1024-byte aligned)   [61,64) swizzle
BWG_HD uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                               uint32_t swizzle) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle & 7u) << 61);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile whose
// rows are 128 bytes and which TMA wrote with 128-byte swizzle: the chunk index
// is XOR-ed with the row index modulo 8 ("GEMM优化（三）", section 2.1).
BWG_HD uint32_t swizzle128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Grouped raster order of output tiles ("GEMM优化（三）", section 3.2-3.4):
// tiles are taken in groups of `group_m` tile rows; inside a group the row
// index runs fastest, so the tiles in flight at one time share a few B column
// strips and `group_m` A row strips, which then stay in L2.
BWG_HD void raster_tile(int t, int num_m_tiles, int num_n_tiles, int group_m, int* m_tile,
                        int* n_tile) {
  const int gsz = group_m * num_n_tiles;
  const int grp = t / gsz;
  const int first_m = grp * group_m;
  const int rows = (num_m_tiles - first_m) < group_m ? (num_m_tiles - first_m) : group_m;
  const int r = t - grp * gsz;
  *m_tile = first_m + r % rows;
  *n_tile = r / rows;
}

// Wave-quantisation split.  With T output tiles on C persistent workers the
// last wave holds only R = T mod C tiles.  Each of those R tiles can be cut
// into f parts: f = 2 halves along N (the MMA N drops to tile_n/2 in the
// instruction descriptor, the MegaMoE page's dynamic N), or, for tiles of two
// stacked 256-row blocks, f = 4 quarters (row block x column half).  A part is
// not 1/f of a tile's time: these kernels are bound by how fast shared memory
// fills, and a part loads more bytes per FLOP than a whole tile, so part f
// costs cost_f/1000 of a tile (its stage bytes over the whole tile's).  The
// cut that makes the last wave, ceil(f*R/C) parts long, cheapest is taken
// (the smaller f on a tie), none if no cut beats the uncut wave.
// Returns R (0: no cut) and the factor in *f.
BWG_HD int tail_split(int T, int C, int max_f, int cost2, int cost4, int* f) {
  *f = 1;
  if (C <= 0 || T <= 0) return 0;
  const int R = T % C;
  if (R == 0) return 0;
  long long best = 1000;  // the uncut last wave: one tile-time
  for (int cand = 2; cand <= max_f; cand *= 2) {
    const long long waves = (static_cast<long long>(cand) * R + C - 1) / C;
    const long long cost = waves * (cand == 2 ? cost2 : cost4);
    if (cost < best) {
      best = cost;
      *f = cand;
    }
  }
  return *f > 1 ? R : 0;
}

// Part costs (per mille of a tile): 256x256 pair tiles cut in halves load
// 24 of 32 KiB per stage; 512x256 two-consumer tiles load 40 (halves) or 24
// (quarters) of 48 KiB.
constexpr int kCostHalf1 = 750;
constexpr int kCostHalf2 = 833;
constexpr int kCostQuarter2 = 500;

// Stream-K last wave (two-consumer pair kernel): with T tiles of kb k-blocks
// on C pairs, the R = T mod C tiles of the last wave (all T when T < C) can
// be shared out by k-block over all C pairs instead of leaving C - R pairs
// idle ("B200 的 2CTA 怎样调优": a short last wave idles SMs; split-K-like
// sharing pays when K is long).  Each pair then does ceil(R*kb/C) iterations
// of the last wave, plus a fixed cost for writing and summing partial
// accumulators.  Taken when that beats `cut_cost` (thousandths of a tile-time:
// 1000 for an uncut last wave, or the cost of the tail_split cut); returns
// the stream-K tile count (0: not taken) and the most segments one pair's
// k-block range can touch in *segs.
constexpr int kStreamKOverhead = 100;
BWG_HD int streamk_tiles(int T, int C, int kb, int cut_cost, int* segs) {
  *segs = 0;
  if (C <= 0 || T <= 0 || kb < 4) return 0;
  const int R = T % C;
  // every pair needs a non-empty range: a pair counted among a tile's
  // sharers must deliver its partial
  if (R == 0 || static_cast<long long>(R) * kb < C) return 0;
  const long long per = (static_cast<long long>(R) * kb + C - 1) / C;
  const long long cost = per * 1000 / kb + kStreamKOverhead;
  if (cost >= cut_cost) return 0;
  *segs = static_cast<int>((per + kb - 1) / kb) + 1;
  return R;
}

// Two-way form (halves only) for the one-consumer kernels.
BWG_HD int tail_split_count(int T, int C) {
  int f = 1;
  return tail_split(T, C, 2, kCostHalf1, 0, &f);
}

// Unit u of a schedule of T tiles whose last R tiles are cut into f parts:
// the tile index, the part (0 .. f-1, 0 for whole tiles) and the count of
// parts of that tile (1 or f).  Whole tiles come first, then the parts of
// each cut tile in turn.
BWG_HD void unit_part(int u, int T, int R, int f, int* tile, int* part, int* parts) {
  const int full = T - R;
  if (u < full || R == 0) {
    *tile = u;
    *part = 0;
    *parts = 1;
  } else {
    const int v = u - full;
    *tile = full + v / f;
    *part = v % f;
    *parts = f;
  }
}

// Two-way form: tile index, column offset inside the tile and the unit's
// width in columns (tile_n, or tile_n/2 for the halves).
BWG_HD void unit_tile(int u, int T, int R, int tile_n, int* tile, int* col_off, int* width) {
  int part = 0, parts = 1;
  unit_part(u, T, R, 2, tile, &part, &parts);
  *col_off = parts == 1 ? 0 : part * (tile_n / 2);
  *width = parts == 1 ? tile_n : tile_n / 2;
}

// The instruction descriptor with its N field replaced (N a multiple of 16).
BWG_HD uint32_t idesc_with_n(uint32_t idesc, uint32_t n) {
  return (idesc & ~(0x3Fu << 17)) | ((n >> 3) << 17);
}

// Stream-K split: W = tiles * kb k-block iterations of a tile list shared out
// evenly over C workers; worker i owns iterations [begin(i), begin(i+1)).  A
// tile whose iterations fall to several workers is finished by the last of
// them to arrive, which sums the partial accumulators in worker order.
BWG_HD long long streamk_begin(int i, long long W, int C) {
  return (W * static_cast<long long>(i)) / C;
}

// The worker whose range holds iteration p (0 <= p < W).
BWG_HD int streamk_owner(long long p, long long W, int C) {
  int i = static_cast<int>((p * C) / W);
  if (i >= C) i = C - 1;
  while (i > 0 && streamk_begin(i, W, C) > p) --i;
  while (i + 1 < C && streamk_begin(i + 1, W, C) <= p) ++i;
  return i;
}

// Workers sharing tile t (kb iterations per tile): the first one and how many.
BWG_HD void streamk_tile_workers(int t, int kb, long long W, int C, int* first, int* count) {
  const int a = streamk_owner(static_cast<long long>(t) * kb, W, C);
  const int b = streamk_owner(static_cast<long long>(t + 1) * kb - 1, W, C);
  *first = a;
  *count = b - a + 1;
}

// Grouped (expert) schedule.  From the offsets of groups g0 .. g0+G-1 build
//   prefix[g] = tiles of groups before g (prefix[G] = all tiles),
//   lo[g], hi[g] = the group's row range, clamped into [0, M] and made
//   non-decreasing so that no tile can reach outside A or D.
// Returns true if the offsets honour the contract (first 0, non-decreasing,
// inside [0, M], last == M when g0+G == G_total).
BWG_HD bool grouped_tables(const int* offsets, int g0, int G, int G_total, int M, int num_n_tiles,
                           int tile_m, int* prefix, int* lo, int* hi) {
  bool ok = true;
  int tiles = 0;
  int prev_hi = 0;
  for (int g = 0; g < G; ++g) {
    int a = offsets[g0 + g];
    int b = offsets[g0 + g + 1];
    if (g0 + g == 0 && a != 0) ok = false;
    if (b < a || a < prev_hi || a < 0 || b > M) ok = false;
    a = a < prev_hi ? prev_hi : a;
    a = a > M ? M : (a < 0 ? 0 : a);
    b = b < a ? a : (b > M ? M : b);
    prev_hi = b;
    prefix[g] = tiles;
    lo[g] = a;
    hi[g] = b;
    tiles += ((b - a + tile_m - 1) / tile_m) * num_n_tiles;
  }
  prefix[G] = tiles;
  if (g0 + G == G_total && offsets[G_total] != M) ok = false;
  return ok;
}

#if defined(__CUDACC__)
// The same tables built by the 32 lanes of one warp (G <= 64), for the
// kernels: each lane loads the offsets of groups lane and lane + 32 and the
// lanes combine them with shuffles, instead of one thread walking the groups
// one global load after the other.  Step by step the loop above computes
//   hi[g] = min(M, max(b_g, a_g, hi[g-1])), hi[-1] = 0,
//   lo[g] = min(M, max(a_g, hi[g-1])),
// with a_g, b_g the offsets at g and g+1; so hi[g] is min(M, max(0, the
// running maximum of max(a_j, b_j) over j <= g)), a prefix maximum, and the
// tile counts' prefix a prefix sum.  Every lane returns the same flag.
__device__ __forceinline__ bool grouped_tables_warp(const int* offsets, int g0, int G, int G_total,
                                                     int M, int num_n_tiles, int tile_m, int* prefix,
                                                     int* lo, int* hi) {
  const unsigned full = 0xffffffffu;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  bool bad = false;
  int run_max = 0;  // running maximum over the groups of earlier halves
  int prev_hi = 0;  // hi of the group before this half's first group
  int carry = 0;    // tiles of the groups of earlier halves
  for (int h = 0; h < 2 && h * 32 < G; ++h) {
    const int g = h * 32 + lane;
    const bool in = g < G;
    const int a = in ? offsets[g0 + g] : 0;
    const int b = in ? offsets[g0 + g + 1] : 0;
    int m = in ? (a > b ? a : b) : run_max;  // inclusive prefix maximum of max(a, b)
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(full, m, d);
      if (lane >= d && y > m) m = y;
    }
    if (run_max > m) m = run_max;
    const int hi_g = m < M ? m : M;  // m >= run_max >= 0
    int before = __shfl_up_sync(full, hi_g, 1);
    if (lane == 0) before = prev_hi;
    int lo_g = a > before ? a : before;
    lo_g = lo_g < M ? lo_g : M;
    if (in) {
      if (g0 + g == 0 && a != 0) bad = true;
      if (b < a || a < before || a < 0 || b > M) bad = true;
    }
    const int t = in ? ((hi_g - lo_g + tile_m - 1) / tile_m) * num_n_tiles : 0;
    int incl = t;  // inclusive prefix sum of the tile counts
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(full, incl, d);
      if (lane >= d) incl += y;
    }
    if (in) {
      prefix[g] = carry + incl - t;
      lo[g] = lo_g;
      hi[g] = hi_g;
    }
    carry += __shfl_sync(full, incl, 31);
    run_max = __shfl_sync(full, m, 31);
    prev_hi = __shfl_sync(full, hi_g, 31);
  }
  if (lane == 0) prefix[G] = carry;
  if (g0 + G == G_total && offsets[G_total] != M) bad = true;
  return !__any_sync(full, bad);
}
#endif

// Tile t of the grouped schedule: its group, first row, first column and the
// group's row end.  Inside a group the row tile runs fastest, so the few
// concurrently running tiles of one column strip share that strip of B_g.
BWG_HD void grouped_tile(int t, int G, const int* prefix, const int* lo, const int* hi,
                         int tile_m, int tile_n, int* g_out, int* m0, int* n0, int* row_end) {
  // the last group g with prefix[g] <= t (prefix is non-decreasing, empty
  // groups repeat a value), by bisection: a scan over 32 groups in shared
  // memory took about 1000 clocks between two units of the MMA warp
  int g = 0, top = G - 1;
  while (g < top) {
    const int mid = (g + top + 1) >> 1;
    if (prefix[mid] <= t)
      g = mid;
    else
      top = mid - 1;
  }
  const int r = t - prefix[g];
  const int mt = (hi[g] - lo[g] + tile_m - 1) / tile_m;
  *g_out = g;
  *m0 = lo[g] + (r % mt) * tile_m;
  *n0 = (r / mt) * tile_n;
  *row_end = hi[g];
}

// Rows of a grouped tile at or below which it is computed with swapped
// operands ("MegaMoE …" section 04: the short token side goes on the MMA's N,
// rounded up to 16), instead of a 256-row tile that is mostly padding.
constexpr int kSwapMaxRows = 128;

// Valid rows of a grouped tile if it is computed swapped, else 0.
BWG_HD int grouped_swap_rows(int m0, int row_end, int tile_m) {
  const int rows = row_end - m0 < tile_m ? row_end - m0 : tile_m;
  return rows <= kSwapMaxRows ? rows : 0;
}

}  // namespace bwg
