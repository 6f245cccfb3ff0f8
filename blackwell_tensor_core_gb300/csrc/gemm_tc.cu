// Persistent, warp-specialised BF16/FP16 GEMM on tcgen05 tensor cores (sm_103a).
//
//   D[M,N] = A[M,K] x B[K,N],  A row-major (K-major operand), B row-major
//   (N-major operand), FP32 accumulation in TMEM, BF16/FP16/FP32 output.
//
// Structure (the design the pages walk through, re-derived for this library):
//  - "使用 Warp Specialization 和 Cluster 扩展 GEMM", step 7: one TMA producer
//    warp, one MMA issuer warp, a warpgroup of epilogue warps, joined by four
//    barrier kinds (SMEM full/empty ring, accumulator full/empty) with
//    producer/consumer phases that start opposite.
//  - same page, step 8: a CTA pair computes a 256x256 tile with
//    tcgen05.mma.cta_group::2; each CTA loads its own 128 rows of A and its own
//    128 columns of B; CTA 0's barrier collects both CTAs' TMA bytes; commits
//    reach both CTAs with CTA mask 0b11; the accumulator-empty barrier in CTA 0
//    collects the epilogue arrivals of both CTAs.
//  - "B200 的 2CTA 怎样调优", section 七: two accumulator slots of 128x256 FP32
//    per CTA (512 TMEM columns), so the epilogue of tile p overlaps the MMA of
//    tile p+1.
//  - "GEMM优化（三）", sections 3.2-3.4: a grouped raster order of output tiles
//    so that concurrently running tiles share A row-strips and B column-strips
//    in L2.
//
// Differences from the pages' kernels: B is consumed in its natural [K,N]
// row-major layout as an MN-major operand (the pages store B as [N,K]); the
// epilogue stages 32-row boxes per warp and issues one TMA store per warp, so
// no warpgroup-wide named barrier is needed; each epilogue warp (not thread)
// arrives once on the accumulator-empty barrier; every barrier wait is bounded
// in time and reports a fault word instead of hanging.
#include "layout.h"
#include "params.h"
#include "ptx.cuh"

namespace bwg {
namespace {

constexpr uint32_t kAStageBytes = kRowsPerCta * kBK * 2;  // 16 KiB: 128 rows x 64 K
constexpr uint32_t kBChunkBytes = 64 * kBK * 2;           // 8 KiB: 64 K rows x 64 N

enum : uint32_t { kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2 };
enum : uint32_t {
  kBarFull = 0,
  kBarEmpty = 1,
  kBarAccFull = 2,
  kBarAccEmpty = 3,
  kBarClcFull = 4,   // a cluster-launch-control response has landed
  kBarClcEmpty = 5   // every role of both CTAs has read a response slot
};

// Dynamic (cluster launch control) scheduling: response slots per CTA.  The
// leader's producer asks for the next unit when it starts a unit, so a pair
// holds at most one unit in reserve; the slots only give the slower roles
// (MMA, epilogue) room to read responses later.
constexpr uint32_t kClcSlots = 4;

__device__ __forceinline__ void record_fault(unsigned long long* err, unsigned long long kind,
                                             uint32_t role, uint32_t bar, uint32_t stage,
                                             uint32_t phase) {
  const unsigned long long code = (kind << 56) | (static_cast<unsigned long long>(role) << 48) |
                                  (static_cast<unsigned long long>(bar) << 40) |
                                  (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 16) |
                                  ((stage & 0xFFu) << 8) | (phase & 0xFFu);
  atomicCAS(err, 0ull, code);
}

// One work unit of the cluster: first row (of the pair), first column, its
// width in columns (a whole tile, or half of one in the last wave), the row
// bound for stores (M, or the end of the unit's group) and the group.
struct Tile {
  int m0;
  int n0;
  int width;      // columns of the unit; 0 = nothing to do (second half of a swapped tile)
  int row_end;
  int g;
  int swap_rows;  // > 0: rows m0 .. m0+swap_rows-1 computed with swapped operands
  int cmask;      // MMA consumers with work in this unit (bit c: rows m0 + 256c ..)
  int kb0, kb1;   // k-blocks of the unit (all of K except for stream-K segments)
  int sk;         // stream-K tile index (0 .. sk_tiles-1), or -1
};

// MC pairs per cluster (1, or 2 when the pairs share B through TMA multicast):
// a schedule unit is then a stack of MC tiles along M with the same columns,
// and pair `pair` of the cluster takes tile row (unit row * MC + pair).
// SW (fused SwiGLU): a tile's 256 MMA columns are 128 gate and 128 up
// columns, so it covers 128 output columns; n0 counts output columns.
template <int CG, int MC, bool GROUPED, int NC = 1, bool SW = false, bool DYN = false>
struct Sched {
  static constexpr int kTileM = kRowsPerCta * CG * NC;
  static constexpr int kOutCols = SW ? kTileN / 2 : kTileN;  // output columns of a whole tile
  const GemmParams& p;
  const int* prefix;  // grouped tables in shared memory: prefix[G+1], lo[G], hi[G]
  const int* lo;
  const int* hi;
  int pair;           // this CTA's pair inside the cluster
  int rows_of_units;  // unit rows (tile rows / MC, rounded up)
  int tiles;          // whole tiles
  int split;          // tiles of the last wave that are cut
  int f;              // parts per cut tile (2 halves, or 4 quarters with two consumers)
  int workers;        // pairs (or CTAs) that run at once
  int sk_units;       // stream-K segment units before the data-parallel tiles
  long long sk_iters; // stream-K (tile, k-block) iterations

  __device__ Sched(const GemmParams& p_, const int* prefix_, const int* lo_, const int* hi_,
                   int workers, int pair_)
      : p(p_), prefix(prefix_), lo(lo_), hi(hi_), pair(pair_), workers(workers) {
    rows_of_units = (p.num_m_tiles + MC - 1) / MC;
    if constexpr (GROUPED)
      tiles = prefix[p.G];
    else
      tiles = rows_of_units * p.num_n_tiles;
    f = 1;
    sk_units = 0;
    sk_iters = 0;
    if (kStreamK && p.sk_tiles > 0) {
      // stream-K replaces the last-wave cut
      split = 0;
      sk_units = p.sk_segs * workers;
      sk_iters = static_cast<long long>(p.sk_tiles) * p.num_k_blocks;
    } else {
      split = p.no_tail_split ? 0
                              : tail_split(tiles, workers, NC == 2 ? 4 : 2,
                                           NC == 2 ? kCostHalf2 : kCostHalf1, kCostQuarter2, &f);
    }
  }

  // Stream-K runs only in the dense two-consumer kernel with the static schedule.
  static constexpr bool kStreamK = !GROUPED && MC == 1 && NC == 2 && !SW && !DYN;

  __device__ int total() const {
    if (kStreamK && p.sk_tiles > 0) return sk_units + tiles - p.sk_tiles;
    return tiles - split + split * f;
  }

  // Unit u < sk_units: segment u / workers of pair u % workers's k-block range
  // (empty units have width 0).  The ranges split the sk_tiles * K-blocks
  // iterations of the last sk_tiles tiles evenly, in (tile, k-block) order.
  __device__ Tile at_streamk(int u) const {
    Tile tl;
    const int w = u % workers, j = u / workers;
    const int kb = p.num_k_blocks;
    const long long lo_i = streamk_begin(w, sk_iters, workers);
    const long long hi_i = streamk_begin(w + 1, sk_iters, workers);
    long long pos = lo_i;
    for (int jj = 0; jj < j && pos < hi_i; ++jj) {
      const long long end = (pos / kb + 1) * kb;
      pos = end < hi_i ? end : hi_i;
    }
    tl.swap_rows = 0;
    tl.g = 0;
    tl.row_end = p.M;
    if (pos >= hi_i) {
      tl.width = 0;
      tl.m0 = tl.n0 = tl.kb0 = tl.kb1 = 0;
      tl.sk = -1;
      tl.cmask = 0;
      return tl;
    }
    const long long ts = pos / kb;
    const long long end = (ts + 1) * kb < hi_i ? (ts + 1) * kb : hi_i;
    tl.sk = static_cast<int>(ts);
    tl.kb0 = static_cast<int>(pos - ts * kb);
    tl.kb1 = static_cast<int>(end - ts * kb);
    int mt, nt;
    raster_tile(tiles - p.sk_tiles + tl.sk, rows_of_units, p.num_n_tiles, p.group_m, &mt, &nt);
    tl.m0 = mt * kTileM;
    tl.n0 = nt * kTileN;
    tl.width = kTileN;
    tl.cmask = (tl.m0 + kRowsPerCta * CG < tl.row_end) ? 3 : 1;
    return tl;
  }

  __device__ Tile at(int u) const {
    if constexpr (kStreamK) {
      if (p.sk_tiles > 0) {
        if (u < sk_units) return at_streamk(u);
        u -= sk_units;  // data-parallel tiles: raster order, all but the last sk_tiles
      }
    }
    Tile tl;
    tl.kb0 = 0;
    tl.kb1 = p.num_k_blocks;
    tl.sk = -1;
    int t, part, parts;
    unit_part(u, tiles, split, f, &t, &part, &parts);
    int col_off = parts == 1 ? 0 : (part & 1) * (kOutCols / 2);
    tl.width = parts == 1 ? kTileN : kTileN / 2;
    tl.swap_rows = 0;
    if constexpr (GROUPED) {
      grouped_tile(t, p.G, prefix, lo, hi, kTileM, kOutCols, &tl.g, &tl.m0, &tl.n0, &tl.row_end);
      if constexpr (CG == 2 && NC == 1 && !SW) {
        if (p.swap_ends) tl.swap_rows = grouped_swap_rows(tl.m0, tl.row_end, kTileM);
        // A swapped tile spans all 256 columns in one unit (its MMA M is the
        // column count): if the last-wave split halved it, the first half
        // does the whole tile and the second half nothing.
        if (tl.swap_rows > 0 && tl.width != kTileN) tl.width = (col_off == 0) ? kTileN : 0;
        if (tl.swap_rows > 0) col_off = 0;
      }
    } else {
      int mt, nt;
      raster_tile(t, rows_of_units, p.num_n_tiles, (p.group_m + MC - 1) / MC, &mt, &nt);
      tl.m0 = (mt * MC + pair) * kTileM;
      tl.n0 = nt * kTileN;
      tl.row_end = p.M;
      tl.g = 0;
    }
    tl.n0 += col_off;
    tl.cmask = 1;
    if constexpr (NC == 2) {
      // the second consumer's 256 rows start 256 rows down; skip them if
      // they lie wholly past the end
      tl.cmask = (tl.m0 + kRowsPerCta * CG < tl.row_end) ? 3 : 1;
      if (parts == 4) {  // quarter: one row block, one column half, one consumer
        if (part >> 1) {
          tl.m0 += 2 * kRowsPerCta;
          tl.cmask = (tl.cmask & 2) ? 1 : 0;
        } else {
          tl.cmask &= 1;
        }
      }
      if (tl.cmask == 0) tl.width = 0;
    }
    return tl;
  }
};

// Warp-uniform bounded wait: every lane waits, and the warp proceeds only if
// all lanes saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool ok = mbar_wait(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

template <int CG, bool GROUPED, class PT>
__device__ __forceinline__ const CUtensorMap* b_map(const PT& P, int g) {
  if constexpr (GROUPED)
    return &P.map_b[g];
  else
    return &P.map_b;
}

// SwiGLU of one gate/up accumulator pair: silu(g) * u with
// silu(g) = g * sigmoid(g) = g / (1 + e^-g), using the hardware's
// approximate exponential and reciprocal (a few ulp of FP32, far below the
// final rounding to 16 bits).  For very negative g, e^-g overflows to +inf,
// the reciprocal is 0 and the result a signed zero, the function's limit.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
  return g * rcp_approx(1.0f + __expf(-g)) * u;
}

// NC = MMA consumers per pair (1, or 2 for 512x256 tiles: two A blocks per
// stage share one B stage, each consumer owning half of the TMEM columns).
// SW = fused SwiGLU epilogue ("B200 的 2CTA 怎样调优", section 七,
// Gate/SwiGLU: pair the gate and up column blocks of one GEMM in the
// epilogue).  B is [gate | up] along N; CTA 0 of the pair loads gate columns
// and CTA 1 the matching up columns, so in every CTA's accumulator the first
// half of the MMA columns is gate and the second half up, for the same rows,
// and each epilogue thread finds both values of a pair in its own TMEM lane.
//
// DYN = dynamic scheduling by cluster launch control ("从 CUDA 代码到 GPU
// 执行" section 9; "B200 的 2CTA 怎样调优": with CTA pairs the claim is per
// cluster, so both CTAs get the same unit).  The grid has one cluster per
// unit; a cluster starts with the unit of its own index and, while it works,
// its leader's producer asks the hardware to cancel a cluster that has not
// launched yet and takes over that cluster's unit.  The response is
// multicast into both CTAs; every role reads the responses in order, so the
// producer, MMA and epilogue warps of both CTAs walk the same unit sequence.
template <int CG, int MC, bool GROUPED, int NC, bool SW, bool DYN, class PT>
__device__ void gemm_body(const PT& P, const GemmParams& p) {
  static_assert(!SW || (CG == 2 && MC == 1 && GROUPED), "SwiGLU runs on the grouped pair kernels");
  static_assert(!DYN || (CG == 2 && MC == 1 && NC == 2), "dynamic scheduling: two-consumer pairs");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t crank = (CG == 2) ? cluster_ctarank() : 0u;  // rank in the cluster
  const uint32_t rank = crank & 1u;                             // rank in the CTA pair
  const uint32_t pair = crank >> 1;                             // pair in the cluster (MC == 2)
  const uint32_t leader = crank & ~1u;                          // the pair's MMA-issuing CTA
  const int S = p.stages;
  constexpr uint32_t kBCols = kTileN / CG;             // B columns a CTA loads for a whole tile
  constexpr uint32_t kBStageBytes = kBCols * kBK * 2;  // 32 KiB (1 CTA) or 16 KiB (pair)
  constexpr uint32_t kAStage = NC * kAStageBytes;      // one 128-row A block per consumer
  constexpr uint32_t kEpiWarp0 = NC == 1 ? 2u : 4u;    // first epilogue warp
  constexpr uint32_t kEpiBufs = NC == 1 ? 2u : 1u;     // staging boxes per epilogue warp

  const uint32_t smem_a = base;
  const uint32_t smem_b = smem_a + S * kAStage;
  const uint32_t smem_epi = smem_b + S * kBStageBytes;
  const uint32_t smem_bar = smem_epi + (p.direct_store ? 0u : static_cast<uint32_t>(kEpiBytes));
  auto full_bar = [&](int s) { return smem_bar + 8u * s; };
  auto empty_bar = [&](int s) { return smem_bar + 8u * (S + s); };
  auto acc_full_bar = [&](int a) { return smem_bar + 8u * (2 * S + a); };
  auto acc_empty_bar = [&](int a) { return smem_bar + 8u * (2 * S + 2 + a); };
  const uint32_t tmem_slot = smem_bar + 8u * (2 * S + 4);
  const uint32_t tables = tmem_slot + 16u;
  // CLC responses (16 bytes each, 16-byte aligned) and their barriers, after
  // the grouped tables
  const uint32_t clc = (tables + 4u * (3u * kMaxGroupsPerLaunch + 1u) + 15u) & ~15u;
  auto clc_resp = [&](uint32_t s) { return clc + 16u * s; };
  auto clc_full = [&](uint32_t s) { return clc + 16u * kClcSlots + 8u * s; };
  auto clc_empty = [&](uint32_t s) { return clc + 16u * kClcSlots + 8u * (kClcSlots + s); };
  // readers of each response: the producer of each CTA, the leader's MMA
  // threads, and every epilogue warp of both CTAs
  constexpr uint32_t kClcReaders = 2u + NC + 8u * NC;

  // ---- set-up: barriers, grouped tables, TMEM allocation -----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      // one MMA commit per pair and consumer (multicast writes need every pair)
      mbar_init(empty_bar(s), MC * NC);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full_bar(a), 1);
      mbar_init(acc_empty_bar(a), CG * 4);
    }
    if constexpr (DYN) {
      for (uint32_t s = 0; s < kClcSlots; ++s) {
        mbar_init(clc_full(s), 1);
        mbar_init(clc_empty(s), kClcReaders);
      }
    }
    fence_mbarrier_init();
  }
  // Grouped tables live after the barriers, in shared memory (generic pointers).
  int* tab = reinterpret_cast<int*>(smem_raw + (tables - smem_u32(smem_raw)));
  int* t_prefix = tab;
  int* t_lo = tab + kMaxGroupsPerLaunch + 1;
  int* t_hi = t_lo + kMaxGroupsPerLaunch;
  if constexpr (GROUPED) {
    if (warp == 2) {  // a warp with no set-up duty
      const bool ok = grouped_tables_warp(p.group_offsets, p.g_begin, p.G, p.G_total, p.M,
                                          p.num_n_tiles, kRowsPerCta * CG * NC, t_prefix, t_lo, t_hi);
      if (!ok && crank == 0 && lane == 0) record_fault(p.err, kFaultBadOffsets, 0, 0, 0, 0);
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.map_a);
    prefetch_tensormap(&p.map_d);
    if constexpr (!GROUPED) prefetch_tensormap(&p.map_b);
  }
  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ld_shared_u32(tmem_slot);

  const int first = static_cast<int>((CG == 2) ? cluster_id_x() : blockIdx.x);
  const int stride = static_cast<int>((CG == 2) ? num_clusters_x() : gridDim.x);
  // the last-wave cut counts the pairs that run at once: the grid with the
  // static schedule, the co-resident pairs with the dynamic one
  const Sched<CG, MC, GROUPED, NC, SW, DYN> sched(p, t_prefix, t_lo, t_hi,
                                                  DYN ? p.workers : stride, static_cast<int>(pair));
  const int total = sched.total();
  bool aborted = false;

  // Next unit of this CTA's sequence after unit t: t + stride (static), or the
  // unit of response k (dynamic; -1 when no launch was cancelled, which ends
  // the sequence, or when the wait timed out).  `arm` re-arms the slot for its
  // next response (the producer of each CTA does this); `warp_wide`: all 32
  // lanes read the response and lane 0 releases the slot for the warp.
  auto next_unit = [&](int t, uint32_t& k, uint32_t role, bool arm, bool warp_wide) -> int {
    if constexpr (!DYN) {
      return t + stride;
    } else {
      const uint32_t s = k % kClcSlots;
      const uint32_t ph = (k / kClcSlots) & 1u;
      const bool got = warp_wide ? warp_wait(clc_full(s), ph, p.timeout_ns)
                                 : mbar_wait(clc_full(s), ph, p.timeout_ns);
      if (!got) {
        if (!warp_wide || lane == 0) record_fault(p.err, kFaultTimeout, role, kBarClcFull, s, ph);
        aborted = true;
        return -1;
      }
      uint32_t x = 0;
      const bool ok = clc_query(clc_resp(s), &x);
      if (ok && arm) mbar_arrive_expect_tx(clc_full(s), 16);
      if (warp_wide) __syncwarp();
      // relaxed: the response was read into registers (the query consumed
      // the load) before the arrive issues, which is all the slot's next
      // asynchronous write must wait for
      if (!warp_wide || lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(clc_empty(s), leader));
      ++k;
      return ok ? static_cast<int>(x) / CG : -1;
    }
  };

  if constexpr (NC == 2) {
    // Registers move from warpgroup 0 (TMA and MMA issue: loop state and
    // descriptors) to the epilogue warpgroups, which hold a whole 32 x 256
    // accumulator slice (packed to 16 bits) before the hand-back.
    if (warp < 4)
      setmaxnreg_dec<kRegsControl2C>();
    else
      setmaxnreg_inc<kRegsEpilogue2C>();
  }

  if (warp == 0) {
    // ---- TMA producer: one thread streams A and B k-blocks into the ring ----
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t k = 0;  // CLC responses read so far
      int n_traced = 0;
      if constexpr (DYN) {
        for (uint32_t c = 0; c < kClcSlots; ++c) mbar_arrive_expect_tx(clc_full(c), 16);
      }
      for (int t = first; DYN ? t >= 0 : t < total;
           t = next_unit(t, k, kRoleProducer, /*arm=*/true, /*warp_wide=*/false)) {
        if constexpr (DYN) {
          if (rank == 0) {
            // ask for the unit after this one (response k), once its slot is free
            const uint32_t cs = k % kClcSlots;
            const uint32_t cph = ((k / kClcSlots) & 1u) ^ 1u;
            if (!mbar_wait(clc_empty(cs), cph, p.timeout_ns)) {
              record_fault(p.err, kFaultTimeout, kRoleProducer, kBarClcEmpty, cs, cph);
              aborted = true;
              break;
            }
            clc_try_cancel_multicast(clc_resp(cs), clc_full(cs));
          }
        }
        if (t >= total) continue;  // a unit past the end (grid rounding): nothing to load
        const Tile tl = sched.at(t);
        if (tl.width == 0) continue;
        if (p.trace != nullptr && n_traced < kTraceUnits) {
          unsigned long long* r = p.trace + (static_cast<size_t>(blockIdx.x) * kTraceUnits + n_traced) * kTraceWords;
          r[0] = static_cast<unsigned long long>(t);
          r[1] = globaltimer_ns();
          ++n_traced;
        }
        const uint32_t b_cols = static_cast<uint32_t>(tl.width) / CG;  // this CTA's B columns
        const uint32_t b_chunks = b_cols / 64;
        // Swapped tile: A's rows are the MMA's N, split between the pair; each
        // CTA loads only its half of the rounded-up rows, in 8-row boxes.
        // (the whole 128-row box is loaded: fewer, larger requests measured
        // faster than fetching only the rows used)
        const uint32_t half_rows = static_cast<uint32_t>(((tl.swap_rows + 15) & ~15) / 2);
        const uint32_t stage_tx =
            CG * (static_cast<uint32_t>(__popc(tl.cmask)) * kAStageBytes + b_cols * kBK * 2) +
            p.tx_extra;
        const int a_row = tl.swap_rows > 0 ? tl.m0 + static_cast<int>(rank * half_rows)
                                           : tl.m0 + static_cast<int>(rank) * kRowsPerCta;
        // SwiGLU: rank 0 loads gate columns n0.., rank 1 the up columns
        // swiglu_up + n0.. (the same output columns).
        const int b_col = SW ? tl.n0 + static_cast<int>(rank) * p.swiglu_up
                             : tl.n0 + static_cast<int>(rank * b_cols);
        const CUtensorMap* mb = b_map<CG, GROUPED>(P, tl.g);
        // B box j: 64 columns of D x 64 K.  Row-major B [K, N] (MN-major
        // operand) is addressed (column, k); B stored as [N, K] (K-major, the
        // layout of the pages' kernels) is addressed (k, column).
        const bool bk = p.b_kmajor != 0;
        for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.timeout_ns)) {
            record_fault(p.err, kFaultTimeout, kRoleProducer, kBarEmpty, s, ph ^ 1u);
            aborted = true;
            break;
          }
          const uint32_t sa = smem_a + s * kAStage;
          const uint32_t sb = smem_b + s * kBStageBytes;
          const int k0 = kb * kBK;
          if constexpr (CG == 2) {
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), stage_tx);
            const uint32_t fb = mapa_shared(full_bar(s), leader);
#pragma unroll
            for (int c = 0; c < NC; ++c)  // consumer c's rows start 256 rows further
              if ((tl.cmask >> c) & 1)
                tma_load_2d_pair(sa + c * kAStageBytes, &p.map_a, fb, k0, a_row + c * 2 * kRowsPerCta);
            if constexpr (MC == 1) {
              if (!GROUPED && p.b_one_box && b_chunks == 2) {
                // both 64-column chunks in one load
                if (bk)
                  tma_load_2d_pair(sb, &p.map_b1, fb, k0, b_col);
                else
                  tma_load_3d_pair(sb, &p.map_b1, fb, 0, k0, b_col / 64);
              } else {
                for (uint32_t j = 0; j < b_chunks; ++j) {
                  const int c = b_col + 64 * static_cast<int>(j);
                  tma_load_2d_pair(sb + j * kBChunkBytes, mb, fb, bk ? k0 : c, bk ? c : k0);
                }
              }
            } else {
              // The pairs share B: box j of this CTA's columns is fetched once, by
              // pair j, and multicast to the same-rank CTA of every pair; each
              // destination's bytes complete on its own pair leader's barrier.
              const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (rank + 2)));
              for (uint32_t j = pair; j < b_chunks; j += MC) {
                const int c = b_col + 64 * static_cast<int>(j);
                tma_load_2d_pair_mc(sb + j * kBChunkBytes, mb, fb, bk ? k0 : c, bk ? c : k0, mask);
              }
            }
          } else {
            mbar_arrive_expect_tx(full_bar(s), stage_tx);
            tma_load_2d(sa, &p.map_a, full_bar(s), k0, a_row);
            for (uint32_t j = 0; j < b_chunks; ++j) {
              const int c = b_col + 64 * static_cast<int>(j);
              tma_load_2d(sb + j * kBChunkBytes, mb, full_bar(s), bk ? k0 : c, bk ? c : k0);
            }
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
      }
    }
    __syncwarp();
  } else if (warp >= 1 && warp <= static_cast<uint32_t>(NC)) {
    // ---- MMA issuer: one warp of CTA 0 drives the tensor cores -------------
    // The whole warp walks the loop (stage indices and descriptors stay
    // warp-uniform) and one elected lane issues the MMAs and commits.
    // With two consumers, warp 1 + c issues consumer c's MMAs (its A block,
    // the shared B stage) into TMEM columns [256c, 256c + 256).
    // Commit masks: the stage-empty signal must reach every CTA whose shared
    // memory the next loads of that stage write (all pairs when B is
    // multicast); the accumulator-full signal only this pair.
    const uint16_t empty_mask = static_cast<uint16_t>(MC == 2 ? 0xF : 0x3);
    const uint16_t acc_mask = static_cast<uint16_t>(0x3u << (2 * pair));
    const int cons = static_cast<int>(warp) - 1;  // consumer of this warp
    if (rank == 0) {
      int s = 0;
      uint32_t ph = 0;
      int acc = NC == 1 ? 0 : cons;  // accumulator slot: alternating, or the consumer's own
      uint32_t acc_ph = 0;
      uint32_t k = 0;
      for (int t = first; DYN ? t >= 0 : t < total;
           t = next_unit(t, k, kRoleMma, /*arm=*/false, /*warp_wide=*/true)) {
        if (t >= total) continue;
        const Tile tl = sched.at(t);
        if (tl.width == 0) continue;
        if (!((tl.cmask >> cons) & 1)) {
          // No rows for this consumer: still commit once per stage (the
          // stage-empty barrier counts every consumer), after the stage's
          // full phase so the commit lands in the right phase.
          for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
            if (!warp_wait(full_bar(s), ph, p.timeout_ns)) {
              if (lane == 0) record_fault(p.err, kFaultTimeout, kRoleMma, kBarFull, s, ph);
              aborted = true;
              break;
            }
            if (elect_one()) {
              if constexpr (CG == 2)
                mma_commit_pair_mc(empty_bar(s), empty_mask);
              else
                mma_commit_1cta(empty_bar(s));
            }
            __syncwarp();
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (aborted) break;
          continue;
        }
        if (!warp_wait(acc_empty_bar(acc), acc_ph ^ 1u, p.timeout_ns)) {
          if (lane == 0) record_fault(p.err, kFaultTimeout, kRoleMma, kBarAccEmpty, acc, acc_ph ^ 1u);
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * kTileN;
        const bool swapped = tl.swap_rows > 0;
        // Swapped: MMA A = the B boxes (MN-major, 256 columns as M), MMA B =
        // the A rows (K-major, N = rows rounded up to 16).
        const uint32_t idesc =
            swapped ? idesc_with_n(p.idesc_swap, static_cast<uint32_t>((tl.swap_rows + 15) & ~15))
                    : idesc_with_n(p.idesc, static_cast<uint32_t>(tl.width));
        for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
          if (!warp_wait(full_bar(s), ph, p.timeout_ns)) {
            if (lane == 0) record_fault(p.err, kFaultTimeout, kRoleMma, kBarFull, s, ph);
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint64_t a_desc =
              make_smem_desc(smem_a + s * kAStage + cons * kAStageBytes, 16, 1024, kSwizzle128B);
          // MN-major B: 64-column chunks 8 KiB apart (LBO), the next 16 K
          // values 16 rows (2048 bytes) further.  K-major B: 8-row groups 1 KiB
          // apart, the next 16 K values 32 bytes along each row, as for A.
          const bool bk = p.b_kmajor != 0;
          const uint64_t b_desc = make_smem_desc(smem_b + s * kBStageBytes, bk ? 16u : kBChunkBytes,
                                                 1024, kSwizzle128B);
          const uint32_t b_step = bk ? 32u : 2048u;
          if (elect_one()) {
#pragma unroll
            for (uint32_t kk = 0; kk < kBK / 16; ++kk) {
              // K-major A: the next 16 K values are 32 bytes further along
              // each 128-byte row.
              const uint64_t ad = a_desc + ((kk * 32u) >> 4);
              const uint64_t bd = b_desc + ((kk * b_step) >> 4);
              mma_f16<CG>(d_tmem, swapped ? bd : ad, swapped ? ad : bd, idesc,
                          (kb != tl.kb0 || kk != 0) ? 1u : 0u);
            }
            if constexpr (CG == 2)
              mma_commit_pair_mc(empty_bar(s), empty_mask);
            else
              mma_commit_1cta(empty_bar(s));
          }
          __syncwarp();
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        if (elect_one()) {
          if constexpr (CG == 2)
            mma_commit_pair_mc(acc_full_bar(acc), acc_mask);
          else
            mma_commit_1cta(acc_full_bar(acc));
        }
        __syncwarp();
        if constexpr (NC == 1) {
          if (++acc == 2) {
            acc = 0;
            acc_ph ^= 1u;
          }
        } else {
          acc_ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ---- epilogue: TMEM -> registers -> convert -> swizzled SMEM -> TMA -----
    const uint32_t q = warp & 3u;  // TMEM lane quarter this warp may read
    const int cons = NC == 1 ? 0 : static_cast<int>((warp - kEpiWarp0) >> 2);  // accumulator owner
    const uint32_t ebuf = smem_epi + (warp - kEpiWarp0) * kEpiBufs * kEpiBufBytes;
    const uint32_t acc_empty_leader0 =
        (CG == 2) ? mapa_shared(acc_empty_bar(0), leader) : acc_empty_bar(0);
    const bool out32 = p.out_dtype == kOutF32;
    const bool outbf = p.out_dtype == kOutBF16;
    int acc = NC == 1 ? 0 : cons;
    uint32_t acc_ph = 0;
    uint32_t buf = 0;
    uint32_t k = 0;
    int n_traced = 0;
    for (int t = first; DYN ? t >= 0 : t < total;
         t = next_unit(t, k, kRoleEpilogue, /*arm=*/false, /*warp_wide=*/true)) {
      if (t >= total) continue;
      const Tile tl = sched.at(t);
      if (tl.width == 0 || !((tl.cmask >> cons) & 1)) continue;
      const int trace_i = n_traced++;  // same unit order as the producer's records
      if (!warp_wait(acc_full_bar(acc), acc_ph, p.timeout_ns)) {
        if (lane == 0) record_fault(p.err, kFaultTimeout, kRoleEpilogue, kBarAccFull, acc, acc_ph);
        aborted = true;
        break;
      }
      tc_fence_after();
      const bool tracer = p.trace != nullptr && warp == kEpiWarp0 && lane == 0 && trace_i < kTraceUnits;
      unsigned long long* const trec =
          tracer ? p.trace + (static_cast<size_t>(blockIdx.x) * kTraceUnits + trace_i) * kTraceWords : nullptr;
      if (tracer) trec[3] = globaltimer_ns();
      const int row_w = tl.m0 + cons * 2 * kRowsPerCta + static_cast<int>(rank * kRowsPerCta + q * 32u);
      const uint32_t t_acc = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc) * kTileN;
      if (GROUPED && tl.swap_rows > 0) {
        // Swapped tile: TMEM lane = output column, TMEM column = row.  Each
        // thread writes its column down the tile's valid rows; the 32 lanes
        // of a warp write 32 adjacent columns of one row at a time.
        const int col = tl.n0 + static_cast<int>(rank * kRowsPerCta + q * 32u + lane);
        const int npad = (tl.swap_rows + 15) & ~15;
        const int elt = out32 ? 4 : 2;
        for (int c0 = 0; c0 < npad; c0 += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_acc + c0, v);
          tmem_wait_ld();
          if (c0 + 32 >= npad) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader0 + 8u * acc);
          }
          if (col < p.N) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (c0 + j < tl.swap_rows) {
                uint8_t* dst = static_cast<uint8_t*>(p.d_ptr) +
                               (static_cast<size_t>(tl.m0 + c0 + j) * p.ldd + col) * elt;
                const float x = __uint_as_float(v[j]);
                if (out32)
                  *reinterpret_cast<uint32_t*>(dst) = v[j];
                else
                  *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(
                      (outbf ? pack_bf16x2(x, 0.f) : pack_f16x2(x, 0.f)) & 0xFFFFu);
              }
            }
          }
        }
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1u;
        }
        continue;
      }
      const int sub_cols = out32 ? 32 : 64;
      // SwiGLU: the unit's output columns are half its MMA columns (16-bit
      // output only); gate of output column c is TMEM column c, up is
      // TMEM column width/2 + c.
      const int out_cols = SW ? tl.width / 2 : tl.width;
      const int nsub = out_cols / sub_cols;
      // Hand the accumulator back to the MMA warp as soon as its last TMEM
      // read has completed (before the conversion of that last chunk): with
      // two consumers each owns one accumulator, so its next tile's MMAs wait
      // for this.
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader0 + 8u * acc);
        if (tracer) trec[4] = globaltimer_ns();
      };
      // Stream-K segment of a tile shared by several pairs: every sharer
      // writes its partial accumulator slice (this warp's 32 rows x 256 FP32
      // columns) to its slot in the workspace and counts itself in; the last
      // to arrive sums all slots in slot (= pair) order, so the result does
      // not depend on which pair finished last, and stores the tile slice.
      // A slice is laid out [32-column chunk][float4 index][lane] so that each
      // warp-wide 16-byte store or load covers 512 contiguous bytes.
      bool store_slice = true;   // false: a partial that another warp will finish
      const float* fix = nullptr;  // last arriver: this lane's row in slot 0
      int fix_slots = 0;
      if constexpr (decltype(sched)::kStreamK) {
        if (tl.sk >= 0) {
          int first_w = 0, sharers = 1;
          streamk_tile_workers(tl.sk, p.num_k_blocks, sched.sk_iters, sched.workers, &first_w,
                               &sharers);
          if (sharers > 1) {
            const uint32_t slice = (static_cast<uint32_t>(cons) * 2u + rank) * 4u + q;
            constexpr size_t kSliceFloats = 32u * kTileN;
            const size_t slot_stride = 16u * kSliceFloats;
            const float* tile_ws = p.ws + static_cast<size_t>(tl.sk) * p.ws_slots * slot_stride +
                                   slice * kSliceFloats + lane * 4u;
            float* mine = const_cast<float*>(tile_ws) + (first - first_w) * slot_stride;
#pragma unroll 1
            for (int c = 0; c < kTileN / 32; ++c) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(t_acc + c * 32, v);
              tmem_wait_ld();
              if (c == kTileN / 32 - 1) release_acc();
#pragma unroll
              for (int j = 0; j < 8; ++j)
                __stcg(reinterpret_cast<float4*>(mine + (c * 8 + j) * 128),
                       make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
            }
            __threadfence();
            __syncwarp();
            int is_last = 0;
            if (lane == 0) {
              int* cnt = p.ws_counters + tl.sk * 16 + static_cast<int>(slice);
              is_last = atomicAdd(cnt, 1) == sharers - 1 ? 1 : 0;
              if (is_last) *cnt = 0;  // all sharers are in: ready for the next call
            }
            is_last = __shfl_sync(0xffffffffu, is_last, 0);
            if (is_last) {
              __threadfence();
              fix = tile_ws;
              fix_slots = sharers;
            } else {
              store_slice = false;
            }
          }
        }
      }
      // Stage one 32-row x sub_cols sub-tile (packed in pk) and store it.
      auto emit = [&](int sub, const uint32_t (&pk)[32]) __attribute__((always_inline)) {
        const int col0 = tl.n0 + sub * sub_cols;
        if (col0 >= p.N) return;
        const bool whole_box = !p.direct_store && (!GROUPED || (row_w + 32 <= tl.row_end));
        if (whole_box) {
          if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
          __syncwarp();
          const uint32_t sb = ebuf + buf * kEpiBufBytes;
#pragma unroll
          for (uint32_t j = 0; j < 8; ++j)
            st_shared_v4(sb + swizzle128_offset(lane, j), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                         pk[4 * j + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.map_d, sb, col0, row_w);
            bulk_commit_group();
          }
          buf = (buf + 1u) % kEpiBufs;
        } else {
          // Ragged end of a group, or the register-store epilogue: each
          // thread stores its own row (64 or 32 columns), if inside.
          const int row = row_w + static_cast<int>(lane);
          if (row < tl.row_end) {
            const int elt = out32 ? 4 : 2;
            uint8_t* drow = static_cast<uint8_t*>(p.d_ptr) +
                            (static_cast<size_t>(row) * p.ldd + col0) * elt;
            const int ncols = min(sub_cols, p.N - col0);
            if (ncols == sub_cols) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                reinterpret_cast<uint4*>(drow)[j] =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            } else if (out32) {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < ncols) reinterpret_cast<uint32_t*>(drow)[c] = pk[c];
            } else {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c < ncols)
                  reinterpret_cast<uint16_t*>(drow)[c] =
                      static_cast<uint16_t>(pk[c >> 1] >> ((c & 1) * 16));
            }
          }
        }
      };
      // Two consumers: both accumulators of a pair fill at the same time, so
      // the tensor pipe waits until the epilogue hands them back.  For 16-bit
      // output the warp therefore reads its whole 32 x 256 slice out of TMEM
      // first (packed to 16 bits: 128 registers), releases the accumulator,
      // and only then stages and stores it, while the next tile's MMAs run.
      const bool early = NC == 2 && !out32 && fix == nullptr && store_slice;
      if constexpr (NC == 2) {
        if (early) {
          if constexpr (SW) {
            // one TMEM round trip per 64 output columns: gate and up, 128
            // registers in flight
            uint32_t pks[2][32];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              if (sub < nsub) {
                uint32_t g[2][32], u[2][32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  tmem_ld_32x32b_x32(t_acc + sub * 64 + h * 32, g[h]);
                  tmem_ld_32x32b_x32(t_acc + out_cols + sub * 64 + h * 32, u[h]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    const float y0 =
                        swiglu_f32(__uint_as_float(g[h][2 * i]), __uint_as_float(u[h][2 * i]));
                    const float y1 = swiglu_f32(__uint_as_float(g[h][2 * i + 1]),
                                                __uint_as_float(u[h][2 * i + 1]));
                    pks[sub][16 * h + i] = outbf ? pack_bf16x2(y0, y1) : pack_f16x2(y0, y1);
                  }
                }
              }
            }
            release_acc();
#pragma unroll
            for (int sub = 0; sub < 2; ++sub)
              if (sub < nsub) emit(sub, pks[sub]);
          } else {
            // All four 64-column sub-tiles are read and packed (128
            // registers) before the hand-back, two sub-tiles (128 FP32
            // registers in flight) per TMEM round trip; staging sub-tile 0
            // first and holding three measured 0.7 us longer per tile, as its
            // stores slowed the remaining TMEM reads.  Columns past the
            // unit's width are read (they are inside the accumulator) and
            // not stored.
            auto pack = [&](uint32_t lo, uint32_t hi) {
              return outbf ? pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi))
                           : pack_f16x2(__uint_as_float(lo), __uint_as_float(hi));
            };
            auto load_packed2 = [&](int sub, uint32_t (&pa)[32], uint32_t (&pb)[32]) {
              uint32_t v[4][32];
#pragma unroll
              for (int h = 0; h < 4; ++h) tmem_ld_32x32b_x32(t_acc + sub * 64 + h * 32, v[h]);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                pa[i] = pack(v[0][2 * i], v[0][2 * i + 1]);
                pa[16 + i] = pack(v[1][2 * i], v[1][2 * i + 1]);
                pb[i] = pack(v[2][2 * i], v[2][2 * i + 1]);
                pb[16 + i] = pack(v[3][2 * i], v[3][2 * i + 1]);
              }
            };
            uint32_t pk[4][32];
            load_packed2(0, pk[0], pk[1]);
            load_packed2(2, pk[2], pk[3]);
            release_acc();
#pragma unroll
            for (int sub = 0; sub < 4; ++sub)
              if (sub < nsub) emit(sub, pk[sub]);
          }
        }
      }
      for (int sub = 0; store_slice && !early && sub < nsub; ++sub) {
        uint32_t pk[32];
        const bool last = sub == nsub - 1;
        if (fix != nullptr) {
          // sum of the partial slices, slot by slot, 32 columns at a time
          const size_t slot_stride = 16u * 32u * kTileN;
#pragma unroll 1
          for (int h = 0; h < (out32 ? 1 : 2); ++h) {
            float acc_v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc_v[j] = 0.f;
            const int chunk = out32 ? sub : 2 * sub + h;  // 32-column chunk of the slice
#pragma unroll 1
            for (int sl = 0; sl < fix_slots; ++sl) {
              const float* src = fix + sl * slot_stride + chunk * 8 * 128;
              float4 x[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) x[j] = __ldcg(reinterpret_cast<const float4*>(src + j * 128));
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                acc_v[4 * j] += x[j].x;
                acc_v[4 * j + 1] += x[j].y;
                acc_v[4 * j + 2] += x[j].z;
                acc_v[4 * j + 3] += x[j].w;
              }
            }
            if (out32) {
#pragma unroll
              for (int j = 0; j < 32; ++j) pk[j] = __float_as_uint(acc_v[j]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[16 * h + i] = outbf ? pack_bf16x2(acc_v[2 * i], acc_v[2 * i + 1])
                                       : pack_f16x2(acc_v[2 * i], acc_v[2 * i + 1]);
            }
          }
        } else if constexpr (SW) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(t_acc + sub * 64 + h * 32, g);
            tmem_ld_32x32b_x32(t_acc + out_cols + sub * 64 + h * 32, u);
            tmem_wait_ld();
            if (last && h == 1) release_acc();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float y0 = swiglu_f32(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]));
              const float y1 =
                  swiglu_f32(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]));
              pk[16 * h + i] = outbf ? pack_bf16x2(y0, y1) : pack_f16x2(y0, y1);
            }
          }
        } else if (out32) {
          tmem_ld_32x32b_x32(t_acc + sub * 32, pk);
          tmem_wait_ld();
          if (last) release_acc();
        } else {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(t_acc + sub * 64, v0);
          tmem_ld_32x32b_x32(t_acc + sub * 64 + 32, v1);
          tmem_wait_ld();
          if (last) release_acc();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float lo0 = __uint_as_float(v0[2 * i]), hi0 = __uint_as_float(v0[2 * i + 1]);
            const float lo1 = __uint_as_float(v1[2 * i]), hi1 = __uint_as_float(v1[2 * i + 1]);
            pk[i] = outbf ? pack_bf16x2(lo0, hi0) : pack_f16x2(lo0, hi0);
            pk[16 + i] = outbf ? pack_bf16x2(lo1, hi1) : pack_f16x2(lo1, hi1);
          }
        }
        emit(sub, pk);
      }
      if (p.trace != nullptr && warp == kEpiWarp0 && lane == 0 && trace_i < kTraceUnits)
        p.trace[(static_cast<size_t>(blockIdx.x) * kTraceUnits + trace_i) * kTraceWords + 2] = globaltimer_ns();
      if constexpr (NC == 1) {
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1u;
        }
      } else {
        acc_ph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  // ---- teardown -----------------------------------------------------------
  if (__syncthreads_or(aborted ? 1 : 0)) {
    // A wait gave up: give copies already in flight time to land before the
    // shared memory and TMEM they target are released.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) nanosleep_ns(1000);
  }
  tc_fence_before();
  if constexpr (CG == 2)
    cluster_sync_all();
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
}

template <int CG, int MC>
__global__ void __launch_bounds__(kThreads, 1) gemm_dense_kernel(const __grid_constant__ GemmParams p) {
  gemm_body<CG, MC, false, 1, false, false>(p, p);
}

// 512x256 tiles on a pair: warp 0 TMA, warps 1-2 MMA (one per consumer),
// warp 3 idle, warps 4-7 and 8-11 the epilogue of consumer 0 and 1.
// DYN: one cluster per unit, units claimed by cluster launch control.
template <bool DYN>
__global__ void __launch_bounds__(kThreads2C, 1)
    gemm_dense_2c_kernel(const __grid_constant__ GemmParams p) {
  gemm_body<2, 1, false, 2, false, DYN>(p, p);
}

template <bool SW>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_grouped_kernel(const __grid_constant__ GroupedParams p) {
  gemm_body<2, 1, true, 1, SW, false>(p, p.base);
}

// Grouped, two consumers: 512-row units; the second consumer's 256 rows are
// skipped where a group has 256 rows or fewer left.
template <bool SW, bool DYN>
__global__ void __launch_bounds__(kThreads2C, 1)
    gemm_grouped_2c_kernel(const __grid_constant__ GroupedParams p) {
  gemm_body<2, 1, true, 2, SW, DYN>(p, p.base);
}

template <class K, class P>
cudaError_t launch_cluster(K kernel, const P& p, int cg, int grid, size_t smem, cudaStream_t s,
                           int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cg);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// The two-consumer kernels split their registers with setmaxnreg after
// set-up; the epilogue warpgroups' increase only completes if the CTA was
// launched with at least the registers the split hands out.  Checked once
// per kernel from the compiled register count: a smaller allocation would
// leave the increase waiting for registers that never come free, so such a
// kernel is not launched.
template <class K>
bool two_consumer_regs_ok(K kernel) {
  static const bool ok = [kernel] {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess) return false;
    return static_cast<uint32_t>(a.numRegs) * kThreads2C >= kRegsControl2C * 128u + kRegsEpilogue2C * 256u;
  }();
  return ok;
}

template <class K, class P>
cudaError_t launch_two_consumer(K kernel, const P& p, int grid, size_t smem, cudaStream_t s) {
  if (!two_consumer_regs_ok(kernel)) return cudaErrorLaunchOutOfResources;
  return launch_cluster(kernel, p, 2, grid, smem, s, kThreads2C);
}

}  // namespace

cudaError_t launch_gemm_1cta(const GemmParams& p, int grid, size_t smem, cudaStream_t s) {
  return launch_cluster(gemm_dense_kernel<1, 1>, p, 1, grid, smem, s);
}

cudaError_t launch_gemm_2cta(const GemmParams& p, int grid, size_t smem, cudaStream_t s) {
  return launch_cluster(gemm_dense_kernel<2, 1>, p, 2, grid, smem, s);
}

cudaError_t launch_gemm_2cta_mc(const GemmParams& p, int grid, size_t smem, cudaStream_t s) {
  return launch_cluster(gemm_dense_kernel<2, 2>, p, 4, grid, smem, s);
}

cudaError_t launch_gemm_2cta_2c(const GemmParams& p, int grid, size_t smem, cudaStream_t s,
                                bool dynamic) {
  return dynamic ? launch_two_consumer(gemm_dense_2c_kernel<true>, p, grid, smem, s)
                 : launch_two_consumer(gemm_dense_2c_kernel<false>, p, grid, smem, s);
}

cudaError_t launch_grouped_2c(const GroupedParams& p, int grid, size_t smem, cudaStream_t s,
                              bool swiglu, bool dynamic) {
  if (dynamic)
    return swiglu ? launch_two_consumer(gemm_grouped_2c_kernel<true, true>, p, grid, smem, s)
                  : launch_two_consumer(gemm_grouped_2c_kernel<false, true>, p, grid, smem, s);
  return swiglu ? launch_two_consumer(gemm_grouped_2c_kernel<true, false>, p, grid, smem, s)
                : launch_two_consumer(gemm_grouped_2c_kernel<false, false>, p, grid, smem, s);
}

cudaError_t launch_grouped_2cta(const GroupedParams& p, int grid, size_t smem, cudaStream_t s,
                                bool swiglu) {
  return swiglu ? launch_cluster(gemm_grouped_kernel<true>, p, 2, grid, smem, s)
                : launch_cluster(gemm_grouped_kernel<false>, p, 2, grid, smem, s);
}

static int occupancy_clusters(const void* fn, int cg, size_t smem, int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cg), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cg);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int max_active_clusters_gemm_2c(size_t smem) {
  return occupancy_clusters(reinterpret_cast<const void*>(gemm_dense_2c_kernel<false>), 2, smem,
                            kThreads2C);
}

int max_active_clusters_grouped_2c(size_t smem) {
  return occupancy_clusters(reinterpret_cast<const void*>(gemm_grouped_2c_kernel<false, false>), 2,
                            smem, kThreads2C);
}

int max_active_clusters_gemm(int cluster, bool grouped, size_t smem) {
  const void* fn = grouped ? reinterpret_cast<const void*>(gemm_grouped_kernel<false>)
                   : cluster == 4 ? reinterpret_cast<const void*>(gemm_dense_kernel<2, 2>)
                   : cluster == 2 ? reinterpret_cast<const void*>(gemm_dense_kernel<2, 1>)
                                  : reinterpret_cast<const void*>(gemm_dense_kernel<1, 1>);
  return occupancy_clusters(fn, cluster, smem);
}

cudaError_t set_gemm_attributes(size_t smem) {
  const void* fns[] = {reinterpret_cast<const void*>(gemm_dense_kernel<1, 1>),
                       reinterpret_cast<const void*>(gemm_dense_kernel<2, 1>),
                       reinterpret_cast<const void*>(gemm_dense_kernel<2, 2>),
                       reinterpret_cast<const void*>(gemm_dense_2c_kernel<false>),
                       reinterpret_cast<const void*>(gemm_dense_2c_kernel<true>),
                       reinterpret_cast<const void*>(gemm_grouped_kernel<false>),
                       reinterpret_cast<const void*>(gemm_grouped_kernel<true>),
                       reinterpret_cast<const void*>(gemm_grouped_2c_kernel<false, false>),
                       reinterpret_cast<const void*>(gemm_grouped_2c_kernel<true, false>),
                       reinterpret_cast<const void*>(gemm_grouped_2c_kernel<false, true>),
                       reinterpret_cast<const void*>(gemm_grouped_2c_kernel<true, true>)};
  for (const void* fn : fns) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace bwg
