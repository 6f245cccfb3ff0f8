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
// k are contiguous: the MMA's A operand is MN-major, loaded as 64x64 boxes with
// 128-byte swizzle.  A is row-major [M,K]: the MMA's B operand is K-major, one
// box of m_pad rows x 64 K.  The accumulator has TMEM lane = output column and
// TMEM column = row of D, so each epilogue thread owns one output column and
// writes it down the rows of a [m_pad x 64] staging tile, which a TMA store
// then writes to D (rows >= M are clipped by the tensor bounds).  This avoids
// the in-TMEM transpose the page describes: no transpose is needed when the
// staging tile is written column-wise.
//
// Work split: one 128-column tile per CTA step, persistent over tiles, a ring
// of `stages` k-blocks, two accumulator slots.  The path is HBM-bound (B is
// read once, A is re-read from L2 by every CTA).
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

__global__ void __launch_bounds__(kThreads, 1) small_m_kernel(const __grid_constant__ SmallMParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const int S = p.stages;
  const uint32_t at_stage_bytes = static_cast<uint32_t>(p.m_pad) * kBK * 2;  // m_pad rows x 128 B
  const uint32_t stage_bytes = kBtStageBytes + at_stage_bytes;
  const int out_elt = p.out_dtype == kOutF32 ? 4 : 2;
  const uint32_t half_bytes = static_cast<uint32_t>(p.m_pad) * 64u * out_elt;  // [m_pad][64] tile

  const uint32_t smem_bt = base;
  const uint32_t smem_at = smem_bt + S * kBtStageBytes;
  const uint32_t smem_d = (smem_at + S * at_stage_bytes + 1023u) & ~1023u;
  const uint32_t smem_bar = (smem_d + 2u * half_bytes + 15u) & ~15u;
  auto full_bar = [&](int s) { return smem_bar + 8u * s; };
  auto empty_bar = [&](int s) { return smem_bar + 8u * (S + s); };
  auto acc_full_bar = [&](int a) { return smem_bar + 8u * (2 * S + a); };
  auto acc_empty_bar = [&](int a) { return smem_bar + 8u * (2 * S + 2 + a); };
  const uint32_t tmem_slot = smem_bar + 8u * (2 * S + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full_bar(a), 1);
      mbar_init(acc_empty_bar(a), 4);
    }
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.map_bt);
    prefetch_tensormap(&p.map_at);
    prefetch_tensormap(&p.map_d);
  }
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ld_shared_u32(tmem_slot);
  bool aborted = false;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      const uint32_t tx = stage_bytes + p.tx_extra;
      for (int t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x) {
        const int n0 = t * 128;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, p.timeout_ns)) {
            record_fault_small(p.err, 0, 1, s, ph ^ 1u);
            aborted = true;
            break;
          }
          const int k0 = kb * kBK;
          const uint32_t sbt = smem_bt + s * kBtStageBytes;
          mbar_arrive_expect_tx(full_bar(s), tx);
          tma_load_2d(sbt, &p.map_bt, full_bar(s), n0, k0);
          tma_load_2d(sbt + kBtChunkBytes, &p.map_bt, full_bar(s), n0 + 64, k0);
          tma_load_2d(smem_at + s * at_stage_bytes, &p.map_at, full_bar(s), k0, 0);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      for (int t = blockIdx.x; t < p.num_tiles && !aborted; t += gridDim.x) {
        if (!mbar_wait(acc_empty_bar(acc), acc_ph ^ 1u, p.timeout_ns)) {
          record_fault_small(p.err, 1, 3, acc, acc_ph ^ 1u);
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * 256u;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait(full_bar(s), ph, p.timeout_ns)) {
            record_fault_small(p.err, 1, 0, s, ph);
            aborted = true;
            break;
          }
          tc_fence_after();
          // MMA A = B^T tile (MN-major, two 64-channel boxes 8 KiB apart),
          // MMA B = A tile (K-major, 128-byte rows, 8-row groups 1 KiB apart).
          const uint64_t a_desc =
              make_smem_desc(smem_bt + s * kBtStageBytes, kBtChunkBytes, 1024, kSwizzle128B);
          const uint64_t b_desc = make_smem_desc(smem_at + s * at_stage_bytes, 16, 1024, kSwizzle128B);
#pragma unroll
          for (uint32_t kk = 0; kk < kBK / 16; ++kk)
            mma_f16<1>(d_tmem, a_desc + ((kk * 2048u) >> 4), b_desc + ((kk * 32u) >> 4), p.idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          mma_commit_1cta(empty_bar(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        mma_commit_1cta(acc_full_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = output columns.
    const uint32_t q = warp & 3u;
    const uint32_t ch = q * 32u + lane;              // column within the 128-wide tile
    const uint32_t half = ch >> 6;                   // which 64-column staging tile
    const uint32_t col_in_half = ch & 63u;
    const bool out32 = p.out_dtype == kOutF32;
    const bool outbf = p.out_dtype == kOutBF16;
    const bool store_thread = threadIdx.x == 64;     // first epilogue thread issues TMA stores
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      const int n0 = t * 128;
      const bool seen = mbar_wait(acc_full_bar(acc), acc_ph, p.timeout_ns);
      // The four epilogue warps share the staging tile: they go on only if all
      // 128 threads saw the accumulator complete.
      if (!named_bar_and(1, 128, seen)) {
        if (threadIdx.x == 64) record_fault_small(p.err, 2, 2, acc, acc_ph);
        aborted = true;
        break;
      }
      tc_fence_after();
      // The previous tile's TMA store must have finished reading the staging tile.
      if (store_thread) bulk_wait_group_read<0>();
      named_bar_sync(1, 128);
      const uint32_t t_acc = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc) * 256u;
      for (int c0 = 0; c0 < p.m_pad; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_acc + c0, v);
        tmem_wait_ld();
        if (c0 + 32 >= p.m_pad) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_local(acc_empty_bar(acc));
        }
        const int rows = min(32, p.M - c0);
        const uint32_t tile = smem_d + half * half_bytes;
        if (out32) {
#pragma unroll
          for (int r = 0; r < 32; ++r)
            if (r < rows)
              st_shared_u32(tile + (static_cast<uint32_t>(c0 + r) * 64u + col_in_half) * 4u, v[r]);
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            if (r < rows) {
              const float x = __uint_as_float(v[r]);
              const uint32_t h = outbf ? pack_bf16x2(x, 0.f) : pack_f16x2(x, 0.f);
              st_shared_u16(tile + (static_cast<uint32_t>(c0 + r) * 64u + col_in_half) * 2u,
                            static_cast<uint16_t>(h & 0xFFFFu));
            }
          }
        }
      }
      fence_proxy_async_shared();
      named_bar_sync(1, 128);
      if (store_thread) {
        tma_store_2d(&p.map_d, smem_d, n0, 0);
        if (n0 + 64 < p.N) tma_store_2d(&p.map_d, smem_d + half_bytes, n0 + 64, 0);
        bulk_commit_group();
      }
      if (++acc == 2) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
    if (store_thread) bulk_wait_group<0>();
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
  small_m_kernel<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
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
