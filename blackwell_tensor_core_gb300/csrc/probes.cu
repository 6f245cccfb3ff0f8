// Probe kernels: each exercises one hardware mechanism the GEMM kernels rely
// on, in isolation, so that a test can check it against a value the pages
// print or a plain CPU formula:
//  - cluster shared-memory exchange (mapa + ld.shared::cluster + cluster
//    barriers): the two cluster examples of "B200 的 2CTA 怎样调优" (Cluster
//    section: block i of a 2-block cluster reads its peer's marker, giving
//    [1, 0, 3, 2] for 4 blocks) and "从 CUDA 代码到 GPU 执行" (pair_sum: inputs
//    0..7 give [1, 1, 5, 5, 9, 9, 13, 13]);
//  - a TMA load with 128-byte swizzle, whose shared-memory image is compared
//    with the XOR formula of "GEMM优化（三）" section 2.1 (the library's
//    swizzle128_offset);
//  - one tile of tcgen05.mma (M = 128, N = 256, K = 16 per instruction, 1..4
//    instructions) from TMA-loaded operands with the library's descriptors,
//    TMEM allocation and tcgen05.ld read-back, compared with an exact product.
//  - the grouped kernels' warp-parallel schedule tables (grouped_tables_warp),
//    compared with the one-thread loop that defines them.
// They are test hooks: nothing on the GEMM path calls them.  Every wait is
// bounded and reports through the device error word.
#include "layout.h"
#include "params.h"
#include "ptx.cuh"

namespace bwg {
namespace {

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32)
    probe_cluster_pair_kernel(const float* in, float* sum_out, int* peer_out) {
  __shared__ uint32_t marker;
  __shared__ float value;
  if (threadIdx.x == 0) {
    marker = blockIdx.x;
    value = in[blockIdx.x];
  }
  cluster_sync_all();  // both CTAs have written their shared variables
  if (threadIdx.x == 0) {
    const uint32_t peer = cluster_ctarank() ^ 1u;
    const uint32_t peer_marker = ld_shared_cluster_u32(mapa_shared(smem_u32(&marker), peer));
    const uint32_t peer_value = ld_shared_cluster_u32(mapa_shared(smem_u32(&value), peer));
    peer_out[blockIdx.x] = static_cast<int>(peer_marker);
    sum_out[blockIdx.x] = value + __uint_as_float(peer_value);
  }
  cluster_sync_all();  // no CTA leaves while its peer may still read it
}

// One 64 x 64 BF16 box (8 KiB, 128-byte rows) loaded by TMA with 128-byte
// swizzle; the raw shared-memory bytes are copied out.
__global__ void __launch_bounds__(128)
    probe_tma_swizzle_kernel(const __grid_constant__ CUtensorMap map, uint8_t* out,
                             unsigned long long* err, unsigned long long timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_storage;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, 8192);
    tma_load_2d(base, &map, bar, 0, 0);
  }
  ok = mbar_wait(bar, 0, timeout_ns);
  if (!ok && threadIdx.x == 0) atomicCAS(err, 0ull, (kFaultTimeout << 56) | (3ull << 48));
  if (__syncthreads_or(ok ? 0 : 1)) {
    // give a late copy time to land before the block's shared memory goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) nanosleep_ns(1000);
    return;
  }
  const uint8_t* src = smem_raw + (base - smem_u32(smem_raw));
  for (uint32_t i = threadIdx.x; i < 8192 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(src)[i];
}

// D[128, 256] (FP32) = A[128, 16*k_steps] x B[16*k_steps, 256]: A [128, 64] and
// B [64, 256] are loaded like one k-block of the one-CTA GEMM (A K-major, one
// 64-column box; B MN-major, four 64-column boxes), then k_steps MMAs of K = 16
// run into a 256-column TMEM accumulator, which 4 warps read back with
// tcgen05.ld (warp w: TMEM lanes 32w .. 32w+31 = rows).
__global__ void __launch_bounds__(128)
    probe_mma_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     float* d, int k_steps, uint32_t idesc, unsigned long long* err,
                     unsigned long long timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sa = base;            // 16 KiB
  const uint32_t sb = base + 16384u;   // 4 x 8 KiB
  const uint32_t load_bar = smem_u32(&bars[0]);
  const uint32_t mma_bar = smem_u32(&bars[1]);
  const uint32_t warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(load_bar, 1);
    mbar_init(mma_bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&tmem_slot), 256);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(load_bar, 16384u + 4u * 8192u);
    tma_load_2d(sa, &map_a, load_bar, 0, 0);
    for (int j = 0; j < 4; ++j) tma_load_2d(sb + 8192u * j, &map_b, load_bar, 64 * j, 0);
    ok = mbar_wait(load_bar, 0, timeout_ns);
    if (ok) {
      tc_fence_after();
      const uint64_t a_desc = make_smem_desc(sa, 16, 1024, kSwizzle128B);
      const uint64_t b_desc = make_smem_desc(sb, 8192, 1024, kSwizzle128B);
      for (int kk = 0; kk < k_steps; ++kk)
        mma_f16<1>(tmem, a_desc + ((kk * 32u) >> 4), b_desc + ((kk * 2048u) >> 4), idesc,
                   kk > 0 ? 1u : 0u);
      mma_commit_1cta(mma_bar);
      ok = mbar_wait(mma_bar, 0, timeout_ns);
    }
    if (!ok) atomicCAS(err, 0ull, (kFaultTimeout << 56) | (4ull << 48));
  }
  if (__syncthreads_or(ok ? 0 : 1)) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) nanosleep_ns(1000);
  } else {
    tc_fence_after();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t row = warp * 32u + lane;
    for (int c = 0; c < 256; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem + ((warp * 32u) << 16) + static_cast<uint32_t>(c), v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) d[row * 256u + c + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, 256);
  }
}

}  // namespace

cudaError_t launch_probe_cluster_pair(const float* in, float* sum_out, int* peer_out, int n,
                                      cudaStream_t s) {
  probe_cluster_pair_kernel<<<n, 32, 0, s>>>(in, sum_out, peer_out);
  return cudaGetLastError();
}

cudaError_t launch_probe_tma_swizzle(const CUtensorMap& map, void* out, unsigned long long* err,
                                     unsigned long long timeout_ns, cudaStream_t s) {
  const int smem = 8192 + 1024;
  probe_tma_swizzle_kernel<<<1, 128, smem, s>>>(map, static_cast<uint8_t*>(out), err, timeout_ns);
  return cudaGetLastError();
}

namespace {
// out: prefix[G+1], lo[G], hi[G], ok: 3G + 2 ints.
__global__ void __launch_bounds__(32) probe_grouped_tables_kernel(const int* offsets, int g0, int G,
                                                                 int G_total, int M, int num_n_tiles,
                                                                 int tile_m, int* out) {
  const bool ok = grouped_tables_warp(offsets, g0, G, G_total, M, num_n_tiles, tile_m, out,
                                      out + G + 1, out + 2 * G + 1);
  if (threadIdx.x == 0) out[3 * G + 1] = ok ? 1 : 0;
}
}  // namespace

cudaError_t launch_probe_grouped_tables(const int* offsets, int g0, int G, int G_total, int M,
                                        int num_n_tiles, int tile_m, int* out, cudaStream_t s) {
  probe_grouped_tables_kernel<<<1, 32, 0, s>>>(offsets, g0, G, G_total, M, num_n_tiles, tile_m, out);
  return cudaGetLastError();
}

cudaError_t launch_probe_mma(const CUtensorMap& map_a, const CUtensorMap& map_b, float* d, int k_steps,
                             uint32_t idesc, unsigned long long* err, unsigned long long timeout_ns,
                             cudaStream_t s) {
  const int smem = 16384 + 4 * 8192 + 1024;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  probe_mma_kernel<<<1, 128, smem, s>>>(map_a, map_b, d, k_steps, idesc, err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace bwg
