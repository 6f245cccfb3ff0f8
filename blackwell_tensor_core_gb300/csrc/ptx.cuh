// Inline-PTX primitives for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM alloc / MMA / commit / ld / fences), cluster ids and barriers.
//
// Each wrapper is written from the public PTX ISA description of the
// instruction.  The pages this library follows describe the same mechanisms:
// "使用 Warp Specialization 和 Cluster 扩展 GEMM" (four barriers, PipelineState,
// TMEM allocation, cta_group::2 commits with a CTA mask) and
// "GEMM优化（三）在消费级Blackwell上" section 4.3 (single-thread TMA issue with
// an mbarrier transaction count).
#pragma once

#include <cstdint>
#include <cuda.h>

#define BWG_DEV __device__ __forceinline__

namespace bwg {

// ---------------------------------------------------------------- ids -----

BWG_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

BWG_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

BWG_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

BWG_DEV uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

BWG_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

BWG_DEV void nanosleep_ns(uint32_t ns) { asm volatile("nanosleep.u32 %0;" ::"r"(ns)); }

// Whole-cluster barrier (every thread of every CTA in the cluster).
BWG_DEV void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Named barrier for a subset of warps (ids 1..15; 0 is __syncthreads).
BWG_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads.
BWG_DEV bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred P, Q;\n\tsetp.ne.u32 P, %3, 0;\n\t"
      "bar.red.and.pred Q, %1, %2, P;\n\tselp.u32 %0, 1, 0, Q;\n\t}"
      : "=r"(out)
      : "r"(id), "r"(nthreads), "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0;
}

// ------------------------------------------------------------ mbarrier -----

BWG_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

BWG_DEV void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

BWG_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

BWG_DEV void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier addressed in the shared::cluster window (own or peer CTA).
BWG_DEV void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// The same arrive without release ordering.  For arrivals that hand back a
// resource whose last use by the arriving warp has already completed in
// registers: a TMEM accumulator after tcgen05.wait::ld (which blocks until the
// reads are done), a response slot after the query that consumed its load.
// Nothing the warp did before needs ordering against what the arrive
// unblocks, and a release at cluster scope waits for every earlier memory
// operation of the warp to be performed: measured on GB300, 1100-1800 SM
// clocks for an epilogue warp (spilled registers, output staging) and
// 2000-5600 for the MMA warp at a unit change, against 25-50 for this form.
BWG_DEV void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
BWG_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}

BWG_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete.  The wait is
// bounded: after `limit_ns` of global time it gives up and returns false so
// that the caller can record the fault and unwind instead of hanging.
BWG_DEV bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Warp-wide bounded wait: every lane waits, and the result is true only if
// all lanes saw the phase complete.
BWG_DEV bool warp_wait_all(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const bool ok = mbar_wait(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// True in one lane of the (converged) warp.  Issuing tcgen05 operations from
// an elected lane of a warp that runs the loop together, rather than from a
// single lane of a diverged warp, keeps their operands warp-uniform.
BWG_DEV bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred)
      :
      : "memory");
  return pred != 0;
}

// ---------------------------------------------------------------- math ----

// Hardware approximate reciprocal (flushes subnormal inputs and results to
// zero; 1/inf = 0).
BWG_DEV float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------ cluster launch control ---
// "从 CUDA 代码到 GPU 执行" section 9 (CLC): a running cluster asks to cancel
// the launch of a cluster that has not started yet; if that succeeds it does
// that cluster's work itself.  The request is asynchronous: its 16-byte
// response lands in shared memory at `resp` and completes 16 transaction
// bytes on the mbarrier `bar`.  With multicast::cluster::all both land at the
// same offsets in every CTA of the cluster, so one thread asks for the pair.
BWG_DEV void clc_try_cancel_multicast(uint32_t resp, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes"
      ".multicast::cluster::all.b128 [%0], [%1];" ::"r"(resp),
      "r"(bar)
      : "memory");
}

// Decode a response in shared memory: whether a launch was cancelled and, if
// so, the x index of the first CTA of the cancelled cluster.
BWG_DEV bool clc_query(uint32_t resp, uint32_t* first_ctaid_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .b128 R;\n\t.reg .pred P;\n\t"
      "ld.shared.b128 R, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 P, R;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, R;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(resp)
      : "memory");
  *first_ctaid_x = x;
  return ok != 0;
}

// ---------------------------------------------------------------- TMA -----

BWG_DEV void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load into this CTA's shared memory, completing bytes on `bar`
// (a barrier of this CTA).
BWG_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                         int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D and 4-D forms of the same load (coordinates innermost first).
BWG_DEV void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                         int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

BWG_DEV void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                         int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// L2 cache policies for the loads below (fraction 1.0 of the accesses).
BWG_DEV uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

BWG_DEV uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

BWG_DEV uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-, 3- and 4-D tiled loads with an L2 cache policy.
BWG_DEV void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0, int32_t c1,
                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

BWG_DEV void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0, int32_t c1,
                              int32_t c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}

BWG_DEV void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0, int32_t c1,
                              int32_t c2, int32_t c3, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
      : "memory");
}

// Same, for a CTA pair: the completing barrier may live in the peer CTA
// (`bar` is a shared::cluster address, e.g. from mapa_shared).
BWG_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                              int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

BWG_DEV void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                              int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Pair form with cluster multicast: the box lands at offset `dst` in every
// CTA of `cta_mask`, and each destination's bytes complete on the barrier at
// offset `bar` in that destination's pair-leader CTA (`bar` addresses a leader).
BWG_DEV void tma_load_2d_pair_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                 int32_t c1, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "h"(cta_mask)
      : "memory");
}

// 2-D tiled store from this CTA's shared memory (bulk-group completion).
BWG_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

BWG_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups still read shared memory.
template <int N>
BWG_DEV void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N bulk groups are incomplete (writes included).
template <int N>
BWG_DEV void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Bulk copy of `bytes` (multiple of 16, 16-byte aligned) from this CTA's
// shared memory to the shared memory of a CTA of the cluster (`dst` and
// `bar` are shared::cluster addresses of that CTA, e.g. from mapa_shared),
// completing the bytes on that CTA's barrier.
BWG_DEV void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

BWG_DEV float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA store, tcgen05.mma operand reads).
BWG_DEV void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- shared -----

BWG_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

BWG_DEV void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

BWG_DEV void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

BWG_DEV uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Load from the shared::cluster window (own or a peer CTA's shared memory,
// an address from mapa_shared).
BWG_DEV uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// ---------------------------------------------------------- conversion ----

// Round-to-nearest-even packs: low 16 bits <- lo, high 16 bits <- hi.
BWG_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

BWG_DEV uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------- tcgen05 ----
// The .cta_group of every tcgen05 instruction in one kernel must agree, so
// each wrapper takes the group size as a template argument.

template <int CG>
BWG_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

template <int CG>
BWG_DEV void tmem_relinquish() {
  if constexpr (CG == 2)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int CG>
BWG_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

BWG_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BWG_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] x B[smem desc], kind::f16 (bf16/fp16 in, fp32 acc).
template <int CG>
BWG_DEV void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                     uint32_t accumulate) {
  if constexpr (CG == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (this CTA) when all prior MMAs of this thread finish.
BWG_DEV void mma_commit_1cta(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Pair form: arrive on the barrier at offset `bar` in every CTA of `cta_mask`.
BWG_DEV void mma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Per-warpgroup register budgets (all four warps of a warpgroup execute the
// same form).  `dec` returns registers to the CTA's pool; `inc` blocks until
// the pool holds enough, so the budgets of all warpgroups must add up to at
// most the registers the CTA was launched with.
template <uint32_t R>
BWG_DEV void setmaxnreg_dec() {
  static_assert(R >= 24 && R <= 256 && R % 8 == 0, "register budget");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
BWG_DEV void setmaxnreg_inc() {
  static_assert(R >= 24 && R <= 256 && R % 8 == 0, "register budget");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

BWG_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Warp-collective TMEM load: lane i of the warp reads TMEM lane (base lane + i),
// 32 consecutive 32-bit columns starting at the address's column.
BWG_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Warp-collective TMEM load of 16 consecutive 32-bit columns (see above).
BWG_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// One FP32 value rounded to nearest even, as the 16 bits of a BF16 / FP16.
BWG_DEV uint16_t cvt_rn_bf16(float x) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return h;
}

BWG_DEV uint16_t cvt_rn_f16(float x) {
  uint16_t h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return h;
}

}  // namespace bwg
