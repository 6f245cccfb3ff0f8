/*
 * bwgemm: half-precision GEMM on one GB300 (sm_103a) -- C ABI.
 *
 * The operation is the dense product D = A x B with BF16 or FP16 inputs and
 * FP32 accumulation ("B200 的 2CTA 怎样调优", section 七: acc = sum over k of
 * A[i,k]*B[k,j], then the epilogue converts acc to the output type), plus the
 * grouped expert product of "MegaMoE … 融合算子解读" (each expert's rows of A
 * times that expert's weight matrix).
 *
 * Common conventions
 *   - All matrices are row-major with element (not byte) leading dimensions:
 *     A[i,k] at A[i*lda + k], B[k,j] at B[k*ldb + j], D[i,j] at D[i*ldd + j].
 *   - A, B and D are DEVICE pointers on the current CUDA device.  The caller
 *     owns every buffer; the library keeps no pointer after the call returns.
 *   - Every base pointer must be 16-byte aligned and every leading dimension
 *     times the element size a multiple of 16 bytes (the TMA engine's rule);
 *     otherwise the call returns BWG_ERR_ALIGNMENT and does nothing.
 *   - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t
 *     passed as void*, NULL = legacy default stream) and the call never
 *     synchronises.  The return value reports host-detectable errors and
 *     launch failures only; faults found by the kernels while running (a
 *     barrier wait that timed out, inconsistent group offsets) are recorded
 *     in a per-process device error word read by bwg_last_device_error().
 *   - There is no CPU fallback: without a usable sm_103a device the calls
 *     return BWG_ERR_CUDA or BWG_ERR_UNSUPPORTED.
 *   - Thread safety: calls may come from several host threads; the internal
 *     tensor-descriptor cache is guarded by a mutex.
 */
#ifndef BWGEMM_H
#define BWGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BWG_OK = 0,
  BWG_ERR_INVALID_ARG = 1, /* null pointer, negative size, ld too small, bad dtype */
  BWG_ERR_ALIGNMENT = 2,   /* pointer or leading dimension breaks the 16-byte rule */
  BWG_ERR_UNSUPPORTED = 3, /* device is not sm_103 / sm_100 family, or size beyond limits */
  BWG_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  BWG_ERR_TIMEOUT = 5,     /* a kernel gave up waiting on a barrier (device error word) */
  BWG_ERR_SCRATCH_LIMIT = 6 /* gemm_bf16_small_m_noalloc: problem too large for its fixed buffer */
} bwg_status;

typedef enum { BWG_OUT_BF16 = 0, BWG_OUT_FP32 = 1, BWG_OUT_FP16 = 2 } bwg_out_dtype;

/*
 * D[M,N] = A[M,K] x B[K,N]; A and B BF16; FP32 accumulation; D in out_dtype.
 * "使用 Warp Specialization 和 Cluster 扩展 GEMM" (steps 7-8) describes the
 * kernel family: TMA producer, tcgen05 MMA issuer and epilogue warps over an
 * mbarrier ring, 256x256 tiles on CTA pairs.  M <= 128 takes the swapped
 * narrow-N kernel of "MegaMoE …" section 04.
 *   lda >= K, ldb >= N, ldd >= N.  M, N or K == 0: M or N == 0 is a no-op;
 *   K == 0 writes D = 0.  Sizes above 2^31-1 elements per dimension are not
 *   supported.  Returns BWG_OK once the work is enqueued.
 *   The small-M kernel may share a tile's k-blocks among several CTAs.  With
 *   few column tiles (at most half the SMs' worth) the CTAs form clusters and
 *   sum their partials in shared memory; with more tiles than SMs and a ragged
 *   last wave they share k-blocks stream-K style through a device workspace
 *   that the library allocates (cudaMalloc) on the first such call on a
 *   stream and keeps, until the process exits, for later calls on that
 *   stream (streams are told apart by their runtime id, so the per-thread
 *   default stream of each host thread has its own).  A call that would have
 *   to grow that workspace while its stream is being captured into a CUDA
 *   graph returns BWG_ERR_UNSUPPORTED: make one eager call of the largest
 *   shape on the stream first, from the host thread that captures.  Callers that must never see the library
 *   allocate can use gemm_bf16_small_m_noalloc below.
 *   The library also holds a TMA-multicast variant of the pair kernel (two
 *   CTA pairs receive every box of B), selected only by the environment
 *   override BWG_FORCE_KERNEL=2cta_mc; it reads only device memory of the
 *   current GPU, and operands anywhere else (host, another GPU, managed
 *   memory) make the call return BWG_ERR_INVALID_ARG before any launch.
 */
bwg_status gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                     int ldd, int out_dtype, void* stream);

/* Same as gemm_bf16 with FP16 inputs. */
bwg_status gemm_fp16(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                     int ldd, int out_dtype, void* stream);

/*
 * Grouped expert product ("MegaMoE … 融合算子解读", expert GEMMs over routed
 * token buckets): for g in [0, G), rows group_offsets[g] .. group_offsets[g+1]-1
 *     D[r, :] = A[r, :] x B[g]     (r in that range)
 *   A: device [M_total, K] BF16, dense (lda = K).
 *   B: HOST array of G device pointers, each [K, N] BF16 row-major (ldb = N).
 *   D: device [M_total, N] BF16, dense (ldd = N).
 *   group_offsets: DEVICE int32 [G+1], group_offsets[0] = 0, non-decreasing,
 *     group_offsets[G] = M_total; empty groups are allowed.  The values are
 *     read by the kernel (no host synchronisation); offsets that break this
 *     contract are clamped into [0, M_total] and reported through the device
 *     error word (kind 2).
 *   M_total is the row count of A and D: the host needs it for the tensor
 *   descriptors because the offsets live on the device.
 *   G may exceed 64; groups are then processed in launches of 64.
 */
bwg_status grouped_gemm_bf16(const void* A, const void* const* B, void* D, const int* group_offsets,
                             int G, int M_total, int N, int K, void* stream);

/* Same as grouped_gemm_bf16 with FP16 inputs and FP16 output. */
bwg_status grouped_gemm_fp16(const void* A, const void* const* B, void* D, const int* group_offsets,
                             int G, int M_total, int N, int K, void* stream);

/*
 * Grouped expert FC1 with the SwiGLU activation fused into the epilogue
 * ("B200 的 2CTA 怎样调优", section 七, Gate/SwiGLU: y = up x SiLU(gate),
 * with gate and up as column blocks of one GEMM, paired in the epilogue;
 * "MegaMoE … 融合算子解读", section 09: FC1's accumulators go through SwiGLU
 * in registers and only the activation is written).  For g in [0, G) and r in
 * group g's rows:
 *     gate = A[r, :] x B[g][:, 0 : N/2],   up = A[r, :] x B[g][:, N/2 : N]
 *     H[r, j] = silu(gate_j) * up_j,       silu(x) = x / (1 + e^-x)
 *   A, group_offsets, G, M_total, K: as for grouped_gemm_bf16.
 *   B: HOST array of G device pointers, each [K, N] BF16 row-major (ldb = N),
 *     the gate projection in columns 0 .. N/2-1, up in N/2 .. N-1.
 *   H: device [M_total, N/2] BF16, dense (ldh = N/2); the gate/up product is
 *     never written to memory.
 *   N must be a multiple of 16 (the up block must start on a 16-byte
 *   boundary), else BWG_ERR_ALIGNMENT.  Accumulation is FP32; silu and the
 *   product are evaluated in FP32 and rounded once to BF16 (nearest even).
 *   K = 0 writes zeros.  Errors as for grouped_gemm_bf16.
 */
bwg_status grouped_gemm_swiglu_bf16(const void* A, const void* const* B, void* H,
                                    const int* group_offsets, int G, int M_total, int N, int K,
                                    void* stream);

/* Same as grouped_gemm_swiglu_bf16 with FP16 inputs and FP16 output. */
bwg_status grouped_gemm_swiglu_fp16(const void* A, const void* const* B, void* H,
                                    const int* group_offsets, int G, int M_total, int N, int K,
                                    void* stream);

/*
 * The same products with B stored transposed, as B[N, K] row-major (ldb >= K):
 *   D[M,N] = A[M,K] x B^T.  This is the layout of the pages' own kernels
 * ("使用 Warp Specialization 和 Cluster 扩展 GEMM" keeps B as (N, K)) and of
 * weights stored [out_features, in_features].  B then enters the tensor cores
 * as a K-major operand, like A; every kernel, tile and schedule of the
 * [K, N] form applies, with the same rules, statuses and results.  For the
 * grouped forms each B[g] is [N, K] with leading dimension K; with SwiGLU,
 * rows 0 .. N/2-1 of B[g] are the gate block and rows N/2 .. N-1 the up block.
 */
bwg_status gemm_bf16_nt(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                        int ldd, int out_dtype, void* stream);
bwg_status gemm_fp16_nt(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                        int ldd, int out_dtype, void* stream);
bwg_status grouped_gemm_bf16_nt(const void* A, const void* const* B, void* D,
                                const int* group_offsets, int G, int M_total, int N, int K,
                                void* stream);
bwg_status grouped_gemm_fp16_nt(const void* A, const void* const* B, void* D,
                                const int* group_offsets, int G, int M_total, int N, int K,
                                void* stream);
bwg_status grouped_gemm_swiglu_bf16_nt(const void* A, const void* const* B, void* H,
                                       const int* group_offsets, int G, int M_total, int N, int K,
                                       void* stream);
bwg_status grouped_gemm_swiglu_fp16_nt(const void* A, const void* const* B, void* H,
                                       const int* group_offsets, int G, int M_total, int N, int K,
                                       void* stream);

/*
 * No-allocation form of gemm_bf16 for small M (M <= 128).  The pages have no
 * counterpart: it exists for callers that cannot let the library call
 * cudaMalloc -- programs that hand all device memory to their own pool
 * allocator up front (a cudaMalloc from the library would then fail or eat
 * into that budget), and latency-critical loops that must not wait on the
 * allocator (cudaMalloc can block the host and synchronise the device).
 * It computes what gemm_bf16 computes (same arguments and
 * rules) with the stream-K small-M kernel, keeping that kernel's partial sums
 * and per-tile counters in one fixed 32 MiB device array inside the library
 * instead of an allocated workspace:
 *   - the array is part of the library's device code: it takes device
 *     memory on a GPU once that code is loaded there, which (with the CUDA
 *     runtime's default lazy loading) is the first call of any bwgemm entry
 *     point on that device, and keeps it until the process exits.  A caller
 *     that hands all free device memory to its own pool should therefore
 *     make that first call before reserving the pool;
 *   - the first call of this entry point on a device looks up the array's
 *     device address (a runtime symbol lookup, with that device current) and
 *     keeps it; make that first call before any stream capture;
 *   - every call shares the array and leaves its contents behind; each call
 *     clears the tile counters it needs (cudaMemsetAsync on `stream`), so
 *     calls on one stream are safe, but calls whose GPU work overlaps (other
 *     streams without ordering) race on the array;
 *   - problems whose partial sums do not fit return BWG_ERR_SCRATCH_LIMIT:
 *     with rows = M rounded up to 16, tiles = ceil(N/128) and S SMs, they
 *     need tiles * sharers * rows * 128 * 4 bytes (at most 32 MiB - 64 KiB),
 *     where sharers <= ceil(S / tiles) + 1 (3 when N = 16384 on 152 SMs),
 *     and at most 16384 tiles; M > 128 returns BWG_ERR_UNSUPPORTED.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 */
bwg_status gemm_bf16_small_m_noalloc(const void* A, const void* B, void* D, int M, int N, int K,
                                     int lda, int ldb, int ldd, int out_dtype, void* stream);

/*
 * End-to-end convenience form of gemm_bf16 for host-resident data: copies
 * A_host [M,K] and B_host [K,N] (dense, BF16, pinned for the copies to run
 * asynchronously) into the caller's device buffers dA, dB, runs the product
 * into dD ([M,N], out_dtype) and copies dD back to D_host.  The work is
 * pipelined over up to 8 row chunks of A and D (whole 512-row tiles, at
 * least 1024 rows): B and A's chunks are copied in on one internal stream,
 * each chunk's product runs on `stream` once its rows have arrived, and its
 * result is copied back on a second internal stream while the next chunk
 * computes.  Everything starts after the work already queued on `stream`,
 * and `stream` completes only after the last copy back, so the caller
 * synchronises `stream` before reading D_host.  The internal streams and
 * events are made on a device's first call and kept; calls from several
 * host threads on one device are serialised while they enqueue.  The
 * library allocates no device memory.  A call that fails after it has queued
 * copies waits for those copies before it returns its error, so the host
 * buffers may be freed or reused as soon as it returns.
 */
bwg_status gemm_bf16_host(const void* A_host, const void* B_host, void* D_host, int M, int N, int K,
                          int out_dtype, void* dA, void* dB, void* dD, void* stream);

/* Human-readable name of a status code (static string). */
const char* bwg_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  *info receives the raw word (0 if no fault):
 *   bits 56..63 kind (1 barrier wait timed out, 2 invalid group offsets),
 *   48..55 role (0 TMA producer, 1 MMA issuer, 2 epilogue),
 *   40..47 barrier (0 stage full, 1 stage empty, 2 accumulator full,
 *   3 accumulator empty), 16..39 block index, 8..15 stage, 0..7 phase.
 * Returns BWG_OK, BWG_ERR_TIMEOUT (kind 1), BWG_ERR_INVALID_ARG (kind 2) or
 * BWG_ERR_CUDA.  After a timeout the output of the faulting call is undefined.
 */
bwg_status bwg_last_device_error(void* stream, unsigned long long* info);

/*
 * Per-process bound on every barrier wait inside the kernels, in
 * nanoseconds (default 2e9).  A wait that exceeds it records a fault and the
 * kernel unwinds instead of hanging.
 */
void bwg_set_watchdog_ns(unsigned long long ns);

/*
 * Probes: small kernels that check one mechanism each, for the tests.  None
 * is on the GEMM path.  All pointers are device pointers; errors as usual,
 * and a wait that times out is reported by bwg_last_device_error.
 *
 * bwg_probe_cluster_pair: n (even) CTAs in clusters of 2; CTA i writes
 *   peer_out[i] = index of its cluster peer and sum_out[i] = in[i] + in[peer],
 *   read from the peer's shared memory (mapa + ld.shared::cluster).  The
 *   pages print [1, 0, 3, 2] for the peer indices of 4 CTAs ("B200 的 2CTA
 *   怎样调优", Cluster section) and [1, 1, 5, 5, 9, 9, 13, 13] for the sums
 *   of inputs 0..7 ("从 CUDA 代码到 GPU 执行", pair_sum).
 * bwg_probe_tma_swizzle: one TMA load of the 64 x 64 16-bit tile `src`
 *   (row-major, 128-byte rows) with 128-byte swizzle; `out` receives the 8 KiB
 *   shared-memory image ("GEMM优化（三）" section 2.1: 16-byte chunk c of row r
 *   lands at r * 128 + ((c ^ (r % 8)) * 16)).
 * bwg_probe_mma: D [128, 256] FP32 = A[:, 0:16k] x B[0:16k, :] for
 *   k = k_steps (1..4) tcgen05.mma instructions of K = 16, with A [128, 64]
 *   and B [64, 256] row-major BF16 (fp16 = 0) or FP16 (fp16 = 1), loaded by
 *   TMA and read back from TMEM, with the GEMM kernels' descriptors.
 * bwg_probe_grouped_tables: the schedule tables of groups g0 .. g0+G-1
 *   (1 <= G <= 64) that the grouped kernels build from the device int32
 *   offsets [G_total + 1] with one warp; `out` (device int32, 3G + 2) gets
 *   the tile prefix [G + 1], the clamped row starts [G] and ends [G], and 1
 *   or 0 for whether the offsets honour the contract.  The tables equal those
 *   of the grouped_gemm_* contract's sequential definition.
 */
bwg_status bwg_probe_cluster_pair(const float* in, float* sum_out, int* peer_out, int n,
                                  void* stream);
bwg_status bwg_probe_tma_swizzle(const void* src, void* out, void* stream);
bwg_status bwg_probe_mma(const void* A, const void* B, float* D, int k_steps, int fp16,
                         void* stream);
bwg_status bwg_probe_grouped_tables(const int* offsets, int g0, int G, int G_total, int M,
                                    int num_n_tiles, int tile_m, int* out, void* stream);

/*
 * Test hook: adds `bytes` to the transaction count every stage expects, so
 * the stage barriers can never complete and the watchdog path runs.  0 (the
 * default) in normal use.
 */
void bwg_debug_set_tx_extra(unsigned int bytes);

/*
 * Profiling hook: while `buffer` (device memory, or NULL to switch off) is
 * set, every launch of the dense and grouped pair kernels records, for each
 * CTA b and each of its first 64 work units i, five 64-bit words at
 * buffer[(b * 64 + i) * 5]: the unit's index in the schedule, the global
 * time (ns) when the TMA producer started it, the global time when the
 * first epilogue warp finished it, and when that warp saw the accumulator
 * full and handed it back to the MMA issuer.  The buffer needs
 * grid x 64 x 40 bytes;
 * the caller owns it and reads it after synchronising.  Launches of the
 * small-M kernel through gemm_bf16 / gemm_fp16 record instead eight words per
 * CTA b at buffer[8 * b] (grid x 64 bytes), global times in ns (0: not
 * reached): [0] kernel entry, [1] first stage seen by the MMA issuer, [2] last
 * accumulator committed, [3] epilogue finished, [4] accumulator seen by the
 * epilogue, [5] first TMEM load done, [6] first rows staged, [7] last rows
 * staged (the last three for whole-tile segments).
 */
void bwg_debug_set_trace(void* buffer);

/* ---------------------------------------------------------------------
 * Planner overrides (environment variables, read on every call; for
 * experiments and tests -- the defaults are the measured best):
 *   BWG_FORCE_KERNEL   1cta | 2cta | 2cta_mc | 2cta_2c | small_m: kernel kind
 *   BWG_FORCE_STAGES   ring depth (must fit the shared memory)
 *   BWG_EPILOGUE       direct: pair kernels store D from registers (default tma)
 *   BWG_GROUP_M        tile rows per raster group (default 8)
 *   BWG_SCHED          clc | static: two-consumer scheduling (default: clc for
 *                      grouped, static for dense)
 *   BWG_NO_TAIL_SPLIT  1: no last-wave cut
 *   BWG_STREAMK_DENSE  1: stream-K last wave in the dense two-consumer kernel
 *   BWG_SMALL_M_TILE_N output columns per small-M tile (16..128, default 128)
 *   BWG_SMALL_M_SPLIT  0: no cluster split; F (2..8): that cluster size
 *   BWG_STREAMK        1 / 0: force stream-K on / off in the small-M kernel
 *   BWG_SMALL_M_PAIRS  0: fill the small-M stage ring one stage per load
 *   BWG_SMALL_M_L2HINT small-M L2 policies, bit 1: B^T evict-first, bit 0: A
 *                      evict-last (default 2; 0 with the cluster split)
 *   BWG_GROUPED_1C     1: grouped kernels with one MMA consumer (256-row units)
 *   BWG_GROUPED_SWAP   1: swapped-operand group ends (one-consumer grouped kernel)
 *   BWG_B_ONE_BOX      0: dense pair kernels load a CTA's B stage as two
 *                      64-column boxes (default: one load where N % 64 == 0
 *                      or B is [N, K])
 * ------------------------------------------------------------------- */

/* ---------------------------------------------------------------------
 * Host-only planning and layout helpers (no GPU needed; used by tests).
 * ------------------------------------------------------------------- */

typedef enum {
  BWG_KERNEL_NONE = 0,     /* nothing to launch (empty problem) */
  BWG_KERNEL_ZERO = 1,     /* K == 0: D = 0 */
  BWG_KERNEL_1CTA = 2,     /* 128 x 256 tiles, one CTA each */
  BWG_KERNEL_2CTA = 3,     /* 256 x 256 tiles on CTA pairs (cta_group::2) */
  BWG_KERNEL_SMALL_M = 4,  /* swapped operands, MMA N = M rounded up to 16 */
  BWG_KERNEL_2CTA_MC = 5,  /* two pairs per 4-CTA cluster, B shared by TMA multicast */
  BWG_KERNEL_2CTA_2C = 6   /* 512 x 256 tiles on a pair: two MMA consumers share each B stage */
} bwg_kernel_kind;

typedef struct {
  int kernel;              /* bwg_kernel_kind */
  int tile_m, tile_n, tile_k; /* SMALL_M: tile_m = padded rows, tile_n = output columns per
                                 tile (<= 128; the MMA spans 128) */
  int mma_m, mma_n;        /* shape of one tcgen05.mma (mma_n = padded M for SMALL_M) */
  int stages;              /* SMEM ring depth */
  int tiles;               /* output tiles */
  int k_blocks;            /* ceil(K / tile_k) */
  double coverage;         /* M*N / (tiles * tile_m * tile_n) */
  int smem_input_per_cta;  /* bytes of A+B ring per CTA (stages x stage bytes) */
  int smem_total;          /* dynamic shared memory requested per CTA */
  int grid;                /* CTAs launched for `sm_count` SMs */
  uint32_t tx_bytes;       /* bytes the stage barrier expects per k-block */
  uint32_t idesc;          /* instruction descriptor */
  int units;               /* work units: tiles, plus one more for every last-wave tile
                              split in two along N (see bwg_tail_split) */
  int streamk;             /* SMALL_M: 1 if (tile, k-block) iterations are shared evenly
                              over all CTAs; 2CTA_2C: 1 if the last wave is (see
                              sk_tiles); partial tiles are summed through a workspace
                              that the library allocates per stream */
  int workers;             /* CTA pairs (one-CTA kernel: CTAs) that run at once; the
                              last-wave cut is computed for this many */
  int dynamic;             /* 2CTA_2C: 1 if units are claimed at run time by cluster
                              launch control (grid = 2 x units), 0 for the static
                              persistent schedule (grid = 2 x workers) */
  int sk_tiles;            /* 2CTA_2C: tiles of the last wave shared out by k-block over
                              all pairs (stream-K; streamk = 1), 0 if none */
  int sk_segs;             /* 2CTA_2C stream-K: most segments in one pair's range */
  int split;               /* SMALL_M: CTAs of a cluster that share each tile's k-blocks in
                              equal slices and sum their FP32 partials through
                              distributed shared memory (grid = tiles x split); 1 if
                              none.  Taken when the tiles fill at most half the SMs */
  int staging_in_ring;     /* SMALL_M: 1 if every CTA has one tile (or one slice of one
                              tile), so the output staging tile reuses the stage ring,
                              idle by then, and the ring is one stage deeper */
  int bt_loads;            /* SMALL_M: TMA loads that fill one stage of B^T: 1 (B stored
                              [N, K], or row-major B with N and tile_n multiples of 64,
                              through a 3-D view that takes both 64-channel halves at
                              once) or 2 */
  int pair_loads;          /* SMALL_M: 1 if pairs of ring stages are filled by one load of
                              B^T and one of A (K a multiple of 64, and bt_loads = 1);
                              fewer, larger loads measured faster on GB300 */
} bwg_plan_info;

/*
 * Plans a dense call without touching the GPU.  force_kernel = 0 lets the
 * planner choose; force_stages = 0 picks the deepest ring that fits in
 * shared memory.  sm_count sizes the persistent grid.
 */
bwg_status bwg_plan(int M, int N, int K, int out_dtype, int sm_count, int force_kernel,
                    int force_stages, bwg_plan_info* out);

/* Argument validation exactly as gemm_bf16/gemm_fp16 apply it (host only). */
bwg_status bwg_check_gemm_args(const void* A, const void* B, const void* D, int M, int N, int K,
                               int lda, int ldb, int ldd, int out_dtype);

/* tcgen05 instruction descriptor, kind::f16 with FP32 accumulation
 * (bf16 != 0: BF16 inputs, else FP16; *_mn_major != 0: operand MN-major). */
uint32_t bwg_idesc_f16(int bf16, int a_mn_major, int b_mn_major, int m, int n);

/* tcgen05 shared-memory matrix descriptor (swizzle: 0 none, 2 = 128-byte). */
uint64_t bwg_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes, int swizzle);

/* Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile. */
uint32_t bwg_swizzle128_offset(uint32_t row, uint32_t chunk);

/* Output tile (m_tile, n_tile) processed at linear position t of the
 * grouped raster order used by the dense kernels (host copy of the device
 * scheduler, for tests). */
void bwg_raster_tile(int t, int num_m_tiles, int num_n_tiles, int group_m, int* m_tile,
                     int* n_tile);

/* Host copy of the grouped schedule the grouped kernels run (for tests).
 * offsets: HOST int32 [G+1].  Fills prefix[G+1] (tiles before each group),
 * lo[G], hi[G] (clamped row ranges) for tiles of tile_m rows and 256 columns
 * over N columns; returns 1 if the offsets honour the contract, else 0. */
int bwg_grouped_schedule(const int* offsets, int G, int M_total, int N, int tile_m, int* prefix,
                         int* lo, int* hi);

/* Tile t of that schedule: group, first row, first column, row end. */
void bwg_grouped_tile(int t, int G, const int* prefix, const int* lo, const int* hi, int tile_m,
                      int* g, int* m0, int* n0, int* row_end);

/* Last-wave split of the persistent schedule: with T tiles on C workers,
 * the number of tiles of the last, partly filled wave that are each split in
 * two halves along N (0 when the remainder is more than half a wave). */
int bwg_tail_split(int T, int C);

/* General form: the cut factor f (2 halves, or 4 quarters when max_f is 4,
 * for tiles of two 256-row blocks) that makes the last wave cheapest, where a
 * half of a one-consumer tile costs 0.75 of a tile and a half or quarter of a
 * two-consumer tile 0.833 or 0.5 (their shared-memory bytes per stage);
 * returns the number of cut tiles R (0: none) and stores f. */
int bwg_tail_split_f(int T, int C, int max_f, int* f);
/* Stream-K last wave of the two-consumer kernel (see streamk_tiles in the
   library's scheduler): tiles shared out by k-block, 0 if the last wave
   (costing cut_cost thousandths of a tile-time) is kept; *segs = most
   segments in one pair's k-block range. */
int bwg_streamk_tiles(int T, int C, int kb, int cut_cost, int* segs);

/* Unit u of a schedule whose last R tiles are cut into f parts: tile index,
 * part (0 .. f-1) and parts of that tile (1 or f). */
void bwg_unit_part(int u, int T, int R, int f, int* tile, int* part, int* parts);

/* Unit u of that schedule: tile index, column offset inside the tile and
 * width in columns (tile_n, or tile_n/2 for the split tiles). */
void bwg_unit_tile(int u, int T, int R, int tile_n, int* tile, int* col_off, int* width);

/* Stream-K schedule of the small-M kernel (host copy, for tests): with
 * `tiles` tiles of `kb` k-blocks on C CTAs, the first iteration CTA i owns,
 * and for tile t the first CTA sharing it and how many CTAs share it. */
long long bwg_streamk_begin(int i, long long W, int C);
void bwg_streamk_tile_workers(int t, int kb, long long W, int C, int* first, int* count);

/* Valid rows of a grouped tile starting at row m0 of a group ending at
 * row_end if the grouped kernel computes it with swapped operands (rows up to
 * 128 go on the MMA's N), else 0. */
int bwg_grouped_swap_rows(int m0, int row_end, int tile_m);

/* Library version string (static): "bwgemm <version> (sm_103a) source <hash>",
 * where <hash> is 16 hex digits of SHA-256 over the code of the sources the
 * library was built from (every csrc file and this header, comments and blank
 * space removed), so that a loaded binary can be matched to its sources. */
const char* bwg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BWGEMM_H */
