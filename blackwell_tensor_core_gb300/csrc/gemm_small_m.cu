// Small-M GEMM by operand swap ("swapAB") with a narrow, padded MMA N.
//
//   D[M,N] = A[M,K] x B[K,N] with M <= 128 is computed as D^T = B^T x A^T:
//   the MMA's M dimension (128) runs over output columns n (channels) and its
//   N dimension over the M rows (tokens), padded up to a multiple of 16.
//
// "MegaMoE … 融合算子解读", section 04 (dynamic N and swapAB): put the short,
// irregular token dimension on the MMA's N, which the instruction descriptor
// sets at run time in steps of 16, so the tensor cores skip most padding.
//
// Operands as stored: B is row-major [K,N], so B^T's 128 channel values for one
// k are contiguous: the MMA's A operand is MN-major, two 64-channel x 64-K
// blocks with 128-byte swizzle, taken by one load through a 3-D view of B
// (64 channels, k, channel group).  A is row-major [M,K]: the MMA's B operand
// is K-major, one box of m_pad rows x 64 K.  Measured on GB300, this kernel
// streams B faster the fewer TMA loads it issues per byte: two 64x64 boxes a
// stage ran 8% slower than one 3-D load, and filling two stages per load
// (4-D view of B, 3-D of A) gained up to 8% more, depending on the shape and
// the GPU.  The accumulator has TMEM lane = output column and
// TMEM column = row of D, so each epilogue thread owns one output column and
// writes it down the rows of a [m_pad x 64] staging tile, which a TMA store
// then writes to D (rows >= M are clipped by the tensor bounds).  No transpose
// step is needed when the staging tile is written column-wise.
//
// Work split.  The path is bound by HBM (B is read once).  Two ways keep all
// SMs streaming:
//  - a narrower tile stride: a tile stores tile_n <= 128 output columns (the
//    MMA and the loads still span 128, the extra columns come from L2 since
//    the neighbouring tile reads them at the same time), so N/tile_n tiles
//    fill the SMs while every CTA walks K in step with the others and the
//    CTAs together read whole rows of B from DRAM;
//  - stream-K, when there are more tiles than SMs or far fewer: the
//    (tile, k-block) iterations are shared out evenly over all CTAs; a CTA
//    works through one or more "segments" (a tile and a range of its
//    k-blocks).  A segment that covers a whole tile is stored directly.
// The CTAs sharing a tile each write their FP32 partial accumulator to a
// workspace slot (slot = CTA index - first CTA of the tile), then increment
// the tile's counter; the CTA that brings the counter to the number of
// sharers sums the slots in slot order (deterministic), stores D and resets
// the counter.  No CTA ever waits for another.  With stream-K off, segments
// are whole tiles taken persistently (tile = CTA index + i * grid).
//
// Cluster split (few tiles, split > 1): a cluster of `split` CTAs shares one
// tile's k-blocks in equal slices.  When every CTA of the cluster has
// finished its MMAs, all their stage rings are idle; each CTA writes its FP32
// partial into its own ring and bulk-copies the rows that CTA o finishes
// (rows o*ceil(M/split) ..) into o's ring through distributed shared memory,
// counted on o's barrier; each CTA then sums the `split` partials of its rows
// in rank order and stores them.  The partials never leave the chip and no workspace is needed; CTAs
// of one cluster are co-scheduled, so waiting for one another is safe (the
// waits are bounded all the same).
#include "layout.h"
#include "params.h"
#include "ptx.cuh"

namespace bwg {
namespace {

constexpr uint32_t kBtStageBytes = 128 * kBK * 2;  // 16 KiB: 64 K rows x 128 channels (2 boxes)
constexpr uint32_t kBtChunkBytes = 64 * kBK * 2;   // 8 KiB

__device__ __forceinline__ void record_fault_small(unsigned long long* err, uint32_t role,
                                                   uint32_t bar, uint32_t stage, uint32_t phase) {
  const unsigned long long code = (kFaultTimeout << 56) |
                                  (static_cast<unsigned long long>(role) << 48) |
                                  (static_cast<unsigned long long>(bar) << 40) |
                                  (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 16) |
                                  ((stage & 0xFFu) << 8) | (phase & 0xFFu);
  atomicCAS(err, 0ull, code);
}

// The segments of this CTA, in order.
struct Segments {
  const SmallMParams& p;
  long long W;        // all iterations (stream-K)
  long long lo, hi;   // this CTA's iterations (stream-K)

  __device__ explicit Segments(const SmallMParams& p_) : p(p_) {
    W = static_cast<long long>(p.num_tiles) * p.num_k_blocks;
    lo = streamk_begin(blockIdx.x, W, gridDim.x);
    hi = streamk_begin(blockIdx.x + 1, W, gridDim.x);
  }

  // Segment i: false when there is none.
  __device__ bool get(int i, int* t, int* kb0, int* kb1) const {
    if (p.split > 1) {
      // one slice of one tile: clusters are formed from consecutive CTAs
      if (i > 0) return false;
      const int r = static_cast<int>(blockIdx.x) % p.split;
      *t = static_cast<int>(blockIdx.x) / p.split;
      *kb0 = (p.num_k_blocks * r) / p.split;
      *kb1 = (p.num_k_blocks * (r + 1)) / p.split;
      return true;
    }
    if (!p.streamk) {
      const int tile = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      if (tile >= p.num_tiles) return false;
      *t = tile;
      *kb0 = 0;
      *kb1 = p.num_k_blocks;
      return true;
    }
    long long pos = lo;
    for (int j = 0; j < i && pos < hi; ++j) {
      const long long tile = pos / p.num_k_blocks;
      const long long end = (tile + 1) * p.num_k_blocks;
      pos = end < hi ? end : hi;
    }
    if (pos >= hi) return false;
    const long long tile = pos / p.num_k_blocks;
    const long long end = (tile + 1) * p.num_k_blocks < hi ? (tile + 1) * p.num_k_blocks : hi;
    *t = static_cast<int>(tile);
    *kb0 = static_cast<int>(pos - tile * p.num_k_blocks);
    *kb1 = static_cast<int>(end - tile * p.num_k_blocks);
    return true;
  }
};

__global__ void __launch_bounds__(kThreads, 1) small_m_kernel(const __grid_constant__ SmallMParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int S = p.stages;
  unsigned long long* const trace = p.trace != nullptr ? p.trace + 8u * blockIdx.x : nullptr;
  if (trace != nullptr && threadIdx.x == 0) trace[0] = globaltimer_ns();
  const uint32_t at_stage_bytes = static_cast<uint32_t>(p.m_pad) * kBK * 2;  // m_pad rows x 128 B
  const uint32_t stage_bytes = kBtStageBytes + at_stage_bytes;
  const int out_elt = p.out_dtype == kOutF32 ? 4 : 2;
  const uint32_t half_bytes = static_cast<uint32_t>(p.m_pad) * 64u * out_elt;  // [m_pad][64] tile

  const uint32_t smem_bt = base;
  const uint32_t smem_at = smem_bt + S * kBtStageBytes;
  const uint32_t ring_end = smem_at + S * at_stage_bytes;
  // output staging tile: in the ring when every CTA has a single tile (the
  // ring is idle by the time the epilogue runs), else after it
  const uint32_t smem_d = p.staging_in_ring ? base : ((ring_end + 1023u) & ~1023u);
  const uint32_t smem_bar = p.staging_in_ring ? ((ring_end + 15u) & ~15u)
                                              : ((smem_d + 2u * half_bytes + 15u) & ~15u);
  auto full_bar = [&](int s) { return smem_bar + 8u * s; };
  auto empty_bar = [&](int s) { return smem_bar + 8u * (S + s); };
  auto acc_full_bar = [&](int a) { return smem_bar + 8u * (2 * S + a); };
  auto acc_empty_bar = [&](int a) { return smem_bar + 8u * (2 * S + 2 + a); };
  const uint32_t tmem_slot = smem_bar + 8u * (2 * S + 4);
  const uint32_t last_flag = tmem_slot + 4u;  // "this CTA finishes the tile" broadcast
  const uint32_t ready_bar = tmem_slot + 8u;   // split: every CTA of the cluster has its partial
  const uint32_t recv_bar = tmem_slot + 16u;   // split: the other CTAs' rows have landed here

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full_bar(a), 1);
      mbar_init(acc_empty_bar(a), 4);
    }
    mbar_init(ready_bar, static_cast<uint32_t>(p.split > 1 ? p.split : 1));
    mbar_init(recv_bar, 1);
    fence_mbarrier_init();
    prefetch_tensormap(&p.map_bt);
    prefetch_tensormap(&p.map_at);
    if (p.pair_loads) {
      prefetch_tensormap(&p.map_bt2);
      prefetch_tensormap(&p.map_at2);
    }
    prefetch_tensormap(&p.map_d);
    if (p.tile_n > 64) prefetch_tensormap(&p.map_d2);
  }
  const Segments segs(p);
  bool aborted = false;
  // TMA producer (warp 0, lane 0): walks this CTA's segments k-block by
  // k-block.  It is the thread that initialised the barriers, so it fills
  // the first ring stages before the block-wide barrier below: the first
  // loads are in flight while TMEM is being allocated.
  //
  // Fewer, larger loads stream B faster, so a stage of B^T is one load
  // where the layout allows it, and with pair_loads two stages are filled by
  // one load of B^T and one of A.  The pair completes on the first stage's barrier;
  // the second stage's barrier gets a plain arrival.  The MMA issuer takes
  // the stages in order, so it has waited for the pair's bytes before it
  // reads the second stage.
  struct Producer {
    const SmallMParams& p;
    const Segments& segs;
    uint32_t smem_bt, smem_at, at_stage_bytes, bar0, tx;
    int S, i = 0, kb = 0, kb1 = 0, n0 = 0, s = 0;
    uint64_t pol_a = 0, pol_b = 0;  // L2 policies of the A and B^T loads
    uint32_t ph = 0;
    bool have = false, done = false;
    __device__ void issue(int limit, bool* aborted) {
      for (int n = 0; n < limit && !done && !*aborted;) {
        if (!have) {
          int t, kb0;
          if (!segs.get(i, &t, &kb0, &kb1)) {
            done = true;
            break;
          }
          n0 = t * p.tile_n;
          kb = kb0;
          have = true;
        }
        if (kb >= kb1) {
          have = false;
          ++i;
          continue;
        }
        const uint32_t full = bar0 + 8u * s, empty = bar0 + 8u * (S + s);
        const bool pair = p.pair_loads && (s & 1) == 0 && s + 1 < S && kb + 2 <= kb1;
        bool ok = mbar_wait(empty, ph ^ 1u, p.timeout_ns);
        if (!ok) record_fault_small(p.err, 0, 1, s, ph ^ 1u);
        if (ok && pair) {
          ok = mbar_wait(empty + 8u, ph ^ 1u, p.timeout_ns);
          if (!ok) record_fault_small(p.err, 0, 1, s + 1, ph ^ 1u);
        }
        if (!ok) {
          *aborted = true;
          break;
        }
        const int k0 = kb * kBK;
        const uint32_t sbt = smem_bt + s * kBtStageBytes;
        const uint32_t sat = smem_at + s * at_stage_bytes;
        if (pair) {
          mbar_arrive_expect_tx(full, 2u * (tx - p.tx_extra) + p.tx_extra);
          if (p.b_kmajor)
            tma_load_3d_hint(sbt, &p.map_bt2, full, 0, n0, kb, pol_b);
          else
            tma_load_4d_hint(sbt, &p.map_bt2, full, 0, 0, n0 >> 6, kb, pol_b);
          tma_load_3d_hint(sat, &p.map_at2, full, 0, 0, kb, pol_a);
          mbar_arrive_local(full + 8u);
          if ((s += 2) == S) {
            s = 0;
            ph ^= 1u;
          }
          kb += 2;
          n += 2;
          continue;
        }
        mbar_arrive_expect_tx(full, tx);
        // B^T's 128 channels x 64 K: row-major B [K, N] is addressed
        // (channel, k) or (channel in group, k, group), B stored as [N, K]
        // (k, channel)
        if (p.b_kmajor) {
          tma_load_2d_hint(sbt, &p.map_bt, full, k0, n0, pol_b);
        } else if (p.bt_boxes == 1) {
          tma_load_3d_hint(sbt, &p.map_bt, full, 0, k0, n0 >> 6, pol_b);
        } else {
          tma_load_2d_hint(sbt, &p.map_bt, full, n0, k0, pol_b);
          tma_load_2d_hint(sbt + kBtChunkBytes, &p.map_bt, full, n0 + 64, k0, pol_b);
        }
        tma_load_2d_hint(sat, &p.map_at, full, k0, 0, pol_a);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
        ++kb;
        ++n;
      }
    }
  } producer{p, segs, smem_bt, smem_at, at_stage_bytes, smem_bar, stage_bytes + p.tx_extra, S};
  // B streams through once, so its loads go in as first to evict: the B
  // lines then do not push A (which every CTA reads) and D out of L2.
  // Measured on GB300 at 72x16384x7168: 43.0 -> 40.9 us; at 128 rows
  // 49.1 -> 40.9 us.  A keeps the normal policy (evict-last gained nothing).
  if (threadIdx.x == 0) {
    producer.pol_b = (p.l2hint & 2) ? l2_policy_evict_first() : l2_policy_evict_normal();
    producer.pol_a = (p.l2hint & 1) ? l2_policy_evict_last() : l2_policy_evict_normal();
  }
  if (threadIdx.x == 0) producer.issue(S, &aborted);
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncwarp();
  if (p.split > 1)
    cluster_sync_all();  // the cluster's barriers are initialised before any remote arrival
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ld_shared_u32(tmem_slot);

  if (warp == 0) {
    if (lane == 0) producer.issue(0x7FFFFFFF, &aborted);
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer.  The whole warp walks the loop, so that stage indices and
    // descriptors stay warp-uniform, and one elected lane issues the MMAs and
    // commits.  (Issued from a single lane of a diverged warp, the four small
    // MMAs of a stage took longer than the stage's bytes take to arrive, and
    // that, not memory, set the kernel's streaming rate.)  Two stages filled
    // by one load are issued after one wait: their bytes complete on the
    // first stage's barrier.
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t acc_ph = 0;
    int t, kb0, kb1;
    // MMA A = B^T tile (MN-major, two 64-channel boxes 8 KiB apart, the next
    // 16 K values 16 rows = 2 KiB further); MMA B = A tile (K-major, 128-byte
    // rows, 8-row groups 1 KiB apart, the next 16 K values 32 bytes along each
    // row).  B stored as [N, K]: the MMA A operand is K-major like the B one.
    const uint32_t a_lbo = p.b_kmajor ? 16u : kBtChunkBytes;
    const uint32_t a_step = p.b_kmajor ? 32u : 2048u;
    for (int i = 0; !aborted && segs.get(i, &t, &kb0, &kb1); ++i) {
      if (!warp_wait_all(acc_empty_bar(acc), acc_ph ^ 1u, p.timeout_ns)) {
        if (lane == 0) record_fault_small(p.err, 1, 3, acc, acc_ph ^ 1u);
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * 256u;
      for (int kb = kb0; kb < kb1;) {
        // the producer's choice for this stage: one load for stages s, s+1
        const int n = (p.pair_loads && (s & 1) == 0 && s + 1 < S && kb + 2 <= kb1) ? 2 : 1;
        if (!warp_wait_all(full_bar(s), ph, p.timeout_ns)) {
          if (lane == 0) record_fault_small(p.err, 1, 0, s, ph);
          aborted = true;
          break;
        }
        if (trace != nullptr && lane == 0 && i == 0 && kb == kb0) trace[1] = globaltimer_ns();
        tc_fence_after();
        for (int j = 0; j < n; ++j) {
          const uint32_t sj = static_cast<uint32_t>(s + j);
          const uint64_t a_desc = make_smem_desc(smem_bt + sj * kBtStageBytes, a_lbo, 1024, kSwizzle128B);
          const uint64_t b_desc = make_smem_desc(smem_at + sj * at_stage_bytes, 16, 1024, kSwizzle128B);
          const bool first = kb + j == kb0;
          if (elect_one()) {
#pragma unroll
            for (uint32_t kk = 0; kk < kBK / 16; ++kk)
              mma_f16<1>(d_tmem, a_desc + ((kk * a_step) >> 4), b_desc + ((kk * 32u) >> 4), p.idesc,
                         (!first || kk > 0) ? 1u : 0u);
            mma_commit_1cta(empty_bar(static_cast<int>(sj)));
          }
          __syncwarp();
        }
        kb += n;
        if ((s += n) == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (aborted) break;
      if (elect_one()) mma_commit_1cta(acc_full_bar(acc));
      __syncwarp();
      if (trace != nullptr && lane == 0) trace[2] = globaltimer_ns();
      if (++acc == 2) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = output columns.
    const uint32_t q = warp & 3u;
    const uint32_t ch = q * 32u + lane;              // column within the 128-wide tile
    const uint32_t half = ch >> 6;                   // which staging tile: columns 0-63, 64-127
    const uint32_t col_in_half = ch & 63u;
    const bool stores = static_cast<int>(ch) < p.tile_n;  // column is part of this tile's output
    const uint32_t pitch = half == 0 ? static_cast<uint32_t>(min(64, p.tile_n))
                                     : static_cast<uint32_t>(max(p.tile_n - 64, 1));
    const bool out32 = p.out_dtype == kOutF32;
    const bool outbf = p.out_dtype == kOutBF16;
    const bool store_thread = threadIdx.x == 64;     // first epilogue thread issues TMA stores
    const size_t slot_floats = static_cast<size_t>(p.m_pad) * 128u;
    int acc = 0;
    uint32_t acc_ph = 0;
    int t, kb0, kb1;

    // Rows r0 .. r0+15 of this thread's column (those below M) into the
    // staging tile.  Staging half h is a dense [m_pad][pitch_h] tile, pitch_0 =
    // min(64, tile_n), pitch_1 = tile_n - 64: exactly the box of the TMA store
    // that writes it.  The epilogue runs once per tile with its code fetched
    // cold, so it is kept short: one conversion and one store per value, in a
    // body that the row loops below reuse.
    const uint32_t row_bytes = pitch * static_cast<uint32_t>(out_elt);
    const uint32_t col_addr = smem_d + half * half_bytes + col_in_half * static_cast<uint32_t>(out_elt);
    auto stage16 = [&](int r0, const uint32_t (&v)[16]) {
      if (!stores) return;
      const int n = min(16, p.M - r0);
      const uint32_t a = col_addr + static_cast<uint32_t>(r0) * row_bytes;
      if (out32) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < n) st_shared_u32(a + r * row_bytes, v[r]);
      } else if (outbf) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < n) st_shared_u16(a + r * row_bytes, cvt_rn_bf16(__uint_as_float(v[r])));
      } else {
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < n) st_shared_u16(a + r * row_bytes, cvt_rn_f16(__uint_as_float(v[r])));
      }
    };
    auto store_staged = [&](int n0) {
      fence_proxy_async_shared();
      named_bar_sync(1, 128);
      if (store_thread) {
        tma_store_2d(&p.map_d, smem_d, n0, 0);
        if (p.tile_n > 64 && n0 + 64 < p.N) tma_store_2d(&p.map_d2, smem_d + half_bytes, n0 + 64, 0);
        bulk_commit_group();
      }
    };

    for (int i = 0; segs.get(i, &t, &kb0, &kb1); ++i) {
      const int n0 = t * p.tile_n;
      const bool whole = (kb0 == 0 && kb1 == p.num_k_blocks);
      const bool seen = mbar_wait(acc_full_bar(acc), acc_ph, p.timeout_ns);
      // The four epilogue warps share the staging tile: they go on only if all
      // 128 threads saw the accumulator complete.
      if (!named_bar_and(1, 128, seen)) {
        if (threadIdx.x == 64) record_fault_small(p.err, 2, 2, acc, acc_ph);
        aborted = true;
        break;
      }
      tc_fence_after();
      if (trace != nullptr && store_thread) trace[4] = globaltimer_ns();
      if (p.split > 1) {
        const int F = p.split;
        const uint32_t me = cluster_ctarank();
        const uint32_t t_acc = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc) * 256u;
        const int rpc = (p.M + F - 1) / F;  // rows each CTA finishes
        const int my_rows = max(0, min(rpc, p.M - static_cast<int>(me) * rpc));
        const uint32_t slot_bytes = static_cast<uint32_t>(rpc) * 512u;  // [rpc][128] FP32
        // 1. This CTA's partial is complete: count the rows it will receive,
        //    then tell every CTA of the cluster (itself included).
        if (store_thread) {
          mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(F - 1) * static_cast<uint32_t>(my_rows) * 512u);
          for (int r = 0; r < F; ++r) mbar_arrive_cluster(mapa_shared(ready_bar, static_cast<uint32_t>(r)));
        }
        // 2. When all have, every stage ring of the cluster is idle.
        const bool ready = mbar_wait(ready_bar, 0, p.timeout_ns);
        if (!named_bar_and(1, 128, ready)) {
          if (store_thread) record_fault_small(p.err, 2, 5, 0, 0);
          aborted = true;
          break;
        }
        if (trace != nullptr && store_thread) trace[5] = globaltimer_ns();
        // 3. The partial goes to this CTA's idle ring as [M rows][128] FP32
        //    (a warp writes 128 contiguous bytes of a row); then one thread
        //    bulk-copies rows [o*rpc, o*rpc + rows_o) to slot `me` of each
        //    other CTA o, counted on o's receive barrier.
#pragma unroll 1
        for (int c0 = 0; c0 < p.m_pad; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(t_acc + c0, v);
          tmem_wait_ld();
          const int n = min(16, p.M - c0);
          const uint32_t a = base + static_cast<uint32_t>(c0) * 512u + ch * 4u;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < n) st_shared_u32(a + j * 512u, v[j]);
        }
        fence_proxy_async_shared();
        named_bar_sync(1, 128);
        const uint32_t recv = base + static_cast<uint32_t>(p.m_pad) * 512u;  // F slots of rpc rows
        if (store_thread) {
          for (int o = 0; o < F; ++o) {
            const int rows_o = min(rpc, p.M - o * rpc);
            if (o == static_cast<int>(me) || rows_o <= 0) continue;
            bulk_copy_to_cluster(mapa_shared(recv + me * slot_bytes, static_cast<uint32_t>(o)),
                                 base + static_cast<uint32_t>(o * rpc) * 512u,
                                 static_cast<uint32_t>(rows_o) * 512u,
                                 mapa_shared(recv_bar, static_cast<uint32_t>(o)));
          }
        }
        if (trace != nullptr && store_thread) trace[6] = globaltimer_ns();
        // 4. Wait for the other CTAs' rows of this CTA.
        const bool got = mbar_wait(recv_bar, 0, p.timeout_ns);
        if (!named_bar_and(1, 128, got)) {
          if (store_thread) record_fault_small(p.err, 2, 6, 0, 0);
          aborted = true;
          break;
        }
        if (trace != nullptr && store_thread) trace[7] = globaltimer_ns();
        // 5. Sum the partials in rank order (this CTA's own from its local
        //    copy) and store this CTA's rows of D, four rows at a time so the
        //    shared-memory loads of a row group are independent.
        const int col = n0 + static_cast<int>(ch);
        if (stores && col < p.N) {
          const int r0 = static_cast<int>(me) * rpc;
          const float* own = reinterpret_cast<const float*>(smem_raw + (base - smem_u32(smem_raw))) +
                             static_cast<size_t>(r0) * 128u + ch;
          const float* slots = reinterpret_cast<const float*>(smem_raw + (recv - smem_u32(smem_raw))) + ch;
          const size_t ldd = static_cast<size_t>(p.ldd);
#pragma unroll 1
          for (int r = 0; r < my_rows; r += 4) {
            float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int src = 0; src < F; ++src) {
              const float* q4 = (src == static_cast<int>(me) ? own : slots + static_cast<size_t>(src) * rpc * 128u) +
                                static_cast<size_t>(r) * 128u;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (r + j < my_rows) sum[j] += q4[j * 128];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (r + j < my_rows) {
                const size_t at = static_cast<size_t>(r0 + r + j) * ldd + col;
                if (out32)
                  static_cast<float*>(p.d)[at] = sum[j];
                else
                  static_cast<uint16_t*>(p.d)[at] = outbf ? cvt_rn_bf16(sum[j]) : cvt_rn_f16(sum[j]);
              }
            }
          }
        }
        break;  // a split CTA has one segment
      }
      // The previous TMA store must have finished reading the staging tile.
      if (store_thread) bulk_wait_group_read<0>();
      named_bar_sync(1, 128);
      const uint32_t t_acc = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc) * 256u;
      int first = 0, sharers = 1;
      float* slot = nullptr;
      if (!whole) {
        streamk_tile_workers(t, p.num_k_blocks, segs.W, gridDim.x, &first, &sharers);
        slot = p.ws + (static_cast<size_t>(t) * p.ws_slots + (blockIdx.x - first)) * slot_floats;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < p.m_pad; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(t_acc + c0, v);
        tmem_wait_ld();
        if (trace != nullptr && store_thread && c0 == 0) trace[5] = globaltimer_ns();
        if (c0 + 16 >= p.m_pad) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_local(acc_empty_bar(acc));
        }
        if (whole) {
          stage16(c0, v);
          if (trace != nullptr && store_thread && c0 == 0) trace[6] = globaltimer_ns();
        } else {
          // partial accumulator -> workspace slot, [row][128 columns] FP32
          const int n = min(16, p.M - c0);
          float* dst = slot + static_cast<size_t>(c0) * 128u + ch;
#pragma unroll
          for (int r = 0; r < 16; ++r)
            if (r < n) dst[r * 128] = __uint_as_float(v[r]);
        }
      }
      if (whole) {
        if (trace != nullptr && store_thread) trace[7] = globaltimer_ns();
        store_staged(n0);
      } else {
        // Publish the partial, count it; the last sharer sums all slots.
        __threadfence();
        named_bar_sync(1, 128);
        if (store_thread) {
          const int old = atomicAdd(p.ws_counters + t, 1);
          const uint32_t is_last = (old == sharers - 1) ? 1u : 0u;
          if (is_last) p.ws_counters[t] = 0;  // every sharer has arrived: ready for the next call
          __threadfence();
          st_shared_u32(last_flag, is_last);
        }
        named_bar_sync(1, 128);
        if (ld_shared_u32(last_flag) != 0u) {
          // Sum the slots in slot order, 32 rows at a time: per slot the 32
          // loads of a thread are independent (and coalesced across the
          // warp), so they are all in flight together.
          const float* tile_slots = p.ws + static_cast<size_t>(t) * p.ws_slots * slot_floats;
#pragma unroll 1
          for (int c0 = 0; c0 < p.M; c0 += 32) {
            const int rows = min(32, p.M - c0);
            const float* src = tile_slots + static_cast<size_t>(c0) * 128u + ch;
            float sum[32], cur[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) {
              sum[r] = 0.f;
              cur[r] = (r < rows) ? __ldcg(src + r * 128) : 0.f;
            }
            // Two slots in flight: the next slot's loads are issued before
            // the current one is added.
#pragma unroll 1
            for (int sl = 0; sl < sharers; ++sl) {
              float nxt[32];
              const float* ns = src + static_cast<size_t>(sl + 1) * slot_floats;
              const bool more = sl + 1 < sharers;
#pragma unroll
              for (int r = 0; r < 32; ++r) nxt[r] = (more && r < rows) ? __ldcg(ns + r * 128) : 0.f;
#pragma unroll
              for (int r = 0; r < 32; ++r) {
                sum[r] += cur[r];
                cur[r] = nxt[r];
              }
            }
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              lo[r] = __float_as_uint(sum[r]);
              hi[r] = __float_as_uint(sum[16 + r]);
            }
            stage16(c0, lo);
            if (rows > 16) stage16(c0 + 16, hi);
          }
          store_staged(n0);
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
    // The CTA may exit once the TMA stores have read the staging tile; their
    // global writes complete on their own before the grid is done.
    if (store_thread) {
      bulk_wait_group_read<0>();
      if (trace != nullptr) trace[3] = globaltimer_ns();
    }
    __syncwarp();
  }

  if (__syncthreads_or(aborted ? 1 : 0)) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) nanosleep_ns(1000);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, kTmemCols);
  }
}

__global__ void zero_fill_kernel(uint8_t* d, int rows, int row_bytes, size_t ld_bytes) {
  const size_t total = static_cast<size_t>(rows) * row_bytes;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / row_bytes, c = i % row_bytes;
    d[r * ld_bytes + c] = 0;
  }
}

}  // namespace

cudaError_t launch_small_m(const SmallMParams& p, int grid, size_t smem, cudaStream_t s) {
  if (p.split <= 1) {
    small_m_kernel<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, small_m_kernel, p);
}

int max_active_clusters_small_m(int cluster, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(small_m_kernel), &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_zero_fill(void* d, int rows, int cols, int ld, int elt_bytes, cudaStream_t s) {
  const size_t total = static_cast<size_t>(rows) * cols * elt_bytes;
  if (total == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<size_t>((total + 255) / 256, 4096));
  zero_fill_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t*>(d), rows, cols * elt_bytes,
                                        static_cast<size_t>(ld) * elt_bytes);
  return cudaGetLastError();
}

int max_active_ctas_small_m(size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, small_m_kernel, kThreads, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t set_small_m_attributes(size_t smem) {
  return cudaFuncSetAttribute(small_m_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem));
}

}  // namespace bwg
