// Host runtime and C ABI: argument checks, the planner (kernel, tile, ring
// depth and grid choice), the TMA descriptor cache and the launches.
//
// Planner rules ("B200 的 2CTA 怎样调优", sections 三 and 八): large problems
// take 256x256 tiles on CTA pairs, with the deepest SMEM ring that fits after
// the epilogue's staging buffers; a problem whose M is at most 128 rows would
// waste half or more of a 256-row tile, so it takes the swapped narrow-N
// kernel instead ("MegaMoE …", section 04).  The persistent grid is the number
// of co-resident clusters the occupancy API reports, capped by the tile count.
// Tensor descriptors ("GEMM优化（三）", section 4.2): 2-D tiled maps with
// 128-byte swizzle and 256-byte L2 promotion; out-of-range boxes fill zeros.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/bwgemm.h"
#include "layout.h"
#include "params.h"

namespace bwg {
cudaError_t set_gemm_attributes(size_t smem);
cudaError_t set_small_m_attributes(size_t smem);
}  // namespace bwg

using namespace bwg;

namespace {

// Device error word: one per device per process, written by kernels that
// give up on a barrier wait (see bwg_last_device_error).
__device__ unsigned long long g_device_error_word;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<unsigned> g_tx_extra{0};
std::atomic<unsigned long long*> g_trace{nullptr};  // unit trace buffer (dense and grouped pair kernels)

constexpr int kMaxDevices = 64;
constexpr int kBarrierArea = 2048;  // barriers, TMEM address slot, grouped tables
constexpr int kGroupM = 8;

struct DeviceState {
  bool ready = false;
  bwg_status init_status = BWG_OK;
  int sm_count = 0;
  int max_smem = 0;
  unsigned long long* err = nullptr;
  int clusters_2cta = 0;
  int clusters_mc = 0;  // 4-CTA clusters (two pairs)
  int clusters_2c = 0;  // pairs of the two-consumer kernel
  int clusters_grouped_2c = 0;
  int ctas_1cta = 0;
  int clusters_grouped = 0;
  int clusters_small[kMaxSplit + 1] = {};  // co-resident clusters of F small-M CTAs, F = 2..8
  // host-buffer entry point: copy streams and chunk events, made on first use
  bool host_ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr;
  cudaEvent_t ev_in[8] = {}, ev_out[8] = {};
  std::mutex host_mu;  // one host-buffer call at a time per device enqueues
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

struct MapKey {
  const void* ptr;
  uint64_t dims[4], strides[3];
  uint32_t box[4];
  int rank, dtype, swizzle, device;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    const uint64_t* w = reinterpret_cast<const uint64_t*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(MapKey) / 8; ++i) h = (h ^ w[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// Stream-K workspace of the small-M kernel (and of the opt-in dense stream-K
// last wave), one per (device, stream): FP32 partial accumulators and
// per-tile arrival counters.  Counters are zeroed when the buffer is made and
// every call leaves them at zero again.  A workspace is reused only by calls
// on its own stream, so calls on one stream are ordered; calls on different
// streams use different workspaces.  Streams are told apart by the runtime's
// stream id, not by the handle: the per-thread default stream has one handle
// but a different stream (and id) in each host thread, and a handle of a
// destroyed stream can come back for a new one.  The buffers are allocated
// (cudaMalloc) on the first call that needs them on a stream and grown when a
// later call needs more; they live until the process exits.  Growing them
// while the stream is being captured into a graph is refused
// (BWG_ERR_UNSUPPORTED): make one eager call of the largest shape first, on
// the same stream and from the same host thread.
struct Workspace {
  float* ws = nullptr;
  int* counters = nullptr;
  size_t ws_bytes = 0;
  int n_counters = 0;
};
struct WorkspaceKey {
  int dev;
  unsigned long long stream_id;
  bool operator==(const WorkspaceKey& o) const { return dev == o.dev && stream_id == o.stream_id; }
};
struct WorkspaceKeyHash {
  size_t operator()(const WorkspaceKey& k) const {
    return static_cast<size_t>((k.stream_id * 1099511628211ull) ^ static_cast<unsigned long long>(k.dev));
  }
};
std::unordered_map<WorkspaceKey, Workspace, WorkspaceKeyHash> g_workspaces;

// Stream ids seen by this host thread, by handle: a stream being captured
// into a graph cannot be asked for its id, so a captured call finds its
// workspace through the id recorded at this thread's last eager call on the
// same handle (for the per-thread default stream, this thread's stream).
thread_local std::unordered_map<uintptr_t, unsigned long long> t_stream_ids;

bwg_status get_workspace(cudaStream_t stream, size_t ws_bytes, int n_counters, Workspace* out) {
  int dev = 0;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return BWG_ERR_CUDA;
  }
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  const uintptr_t handle = reinterpret_cast<uintptr_t>(stream);
  unsigned long long sid = 0;
  if (!capturing) {
    if (cudaStreamGetId(stream, &sid) != cudaSuccess) {
      cudaGetLastError();
      return BWG_ERR_CUDA;
    }
    t_stream_ids[handle] = sid;
  } else {
    const auto it = t_stream_ids.find(handle);
    if (it == t_stream_ids.end()) return BWG_ERR_UNSUPPORTED;  // no eager call on this stream yet
    sid = it->second;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[WorkspaceKey{dev, sid}];
  if (w.ws_bytes < ws_bytes || w.n_counters < n_counters) {
    if (capturing) return BWG_ERR_UNSUPPORTED;
    // grow to cover both the old and the new request, so that alternating
    // shapes settle on one buffer instead of reallocating every call
    const size_t wb = std::max(ws_bytes, w.ws_bytes);
    const int nc = std::max(n_counters, w.n_counters);
    if (w.ws != nullptr || w.counters != nullptr) {
      // the old buffers may still be in use by work queued on this stream
      if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return BWG_ERR_CUDA;
      }
      cudaFree(w.ws);
      cudaFree(w.counters);
      w = Workspace();
    }
    if (cudaMalloc(&w.ws, wb) != cudaSuccess ||
        cudaMalloc(&w.counters, static_cast<size_t>(nc) * sizeof(int)) != cudaSuccess ||
        cudaMemsetAsync(w.counters, 0, static_cast<size_t>(nc) * sizeof(int), stream) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(w.ws);
      cudaFree(w.counters);
      w = Workspace();
      return BWG_ERR_CUDA;
    }
    w.ws_bytes = wb;
    w.n_counters = nc;
  }
  *out = w;
  return BWG_OK;
}

// Zero every stream-K arrival counter of this device (after a timeout).
bwg_status clear_workspace_counters() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& kv : g_workspaces) {
    if (kv.first.dev != dev || kv.second.counters == nullptr) continue;
    if (cudaMemset(kv.second.counters, 0, static_cast<size_t>(kv.second.n_counters) * sizeof(int)) !=
        cudaSuccess)
      return BWG_ERR_CUDA;
  }
  return BWG_OK;
}

// Most CTAs that share one tile under the stream-K split.
int streamk_max_sharers(int tiles, int kb, int grid) {
  const long long W = static_cast<long long>(tiles) * kb;
  int most = 1;
  for (int t = 0; t < tiles; ++t) {
    int first = 0, count = 1;
    streamk_tile_workers(t, kb, W, grid, &first, &count);
    most = std::max(most, count);
  }
  return most;
}



// ------------------------------------------------------------ planning -----

// Per-CTA bytes of one ring stage: nc A blocks of 128 rows and this CTA's
// share of the B columns, 64 K deep.
int dense_stage_bytes(int cg, int nc = 1) {
  return nc * kRowsPerCta * kBK * 2 + (kTileN / cg) * kBK * 2;
}

int dense_smem(int cg, int stages, bool direct_store = false, int nc = 1) {
  return 1024 + stages * dense_stage_bytes(cg, nc) + (direct_store ? 0 : kEpiBytes) + kBarrierArea;
}

// Epilogue choice: "tma" (staged boxes + TMA stores) or "direct" (rows stored
// from registers, which frees the staging space for one more ring stage).
bool direct_store_from_env() {
  const char* v = std::getenv("BWG_EPILOGUE");
  return v != nullptr && !std::strcmp(v, "direct");
}

int small_m_pad(int M) { return std::max(16, (M + 15) & ~15); }

int small_m_stage_bytes(int m_pad) { return 128 * kBK * 2 + m_pad * kBK * 2; }

int small_m_staging(int m_pad, int out_dtype) { return 2 * m_pad * 64 * (out_dtype == kOutF32 ? 4 : 2); }

// Dynamic shared memory of the small-M kernel: alignment slack, the stage
// ring, the output staging tile (unless it lives in the ring), barriers.
int small_m_smem(int m_pad, int out_dtype, int stages, bool staging_in_ring = false) {
  return 1024 + stages * small_m_stage_bytes(m_pad) +
         (staging_in_ring ? 0 : 1024 + small_m_staging(m_pad, out_dtype)) + 512;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Whether the small-M kernel loads a stage of row-major B^T as one box of
// the 3-D channel-group view: N must be a multiple of 64 (the groups tile B)
// and so must the tile stride (every tile starts on a group).
bool small_m_one_bt_box(int N, int tile_n, bool b_kmajor) {
  return b_kmajor || (N % 64 == 0 && tile_n % 64 == 0);
}

// Whether it fills its ring two stages per load: the views that take two
// k-blocks at once tile the matrices exactly only when K is a multiple of 64,
// and for row-major B the stage must be one box.  BWG_SMALL_M_PAIRS=0 turns
// it off.
bool small_m_pairs_ok(int N, int K, int tile_n, int stages, bool b_kmajor) {
  const char* v = std::getenv("BWG_SMALL_M_PAIRS");
  if (v != nullptr && v[0] == '0') return false;
  return K % 64 == 0 && stages >= 2 && small_m_one_bt_box(N, tile_n, b_kmajor);
}

int group_m_from_env() {
  const char* v = std::getenv("BWG_GROUP_M");
  const int g = v ? std::atoi(v) : 0;
  return g > 0 ? g : kGroupM;
}

// Scheduling of the two-consumer kernels: units claimed at run time with
// cluster launch control, or the persistent round-robin loop.  Measured on
// GB300: the grouped FC1 runs 5% faster dynamic (expert units differ in
// cost), dense squares the same either way, so the default is dynamic for
// grouped and static for dense.  BWG_SCHED=clc / static overrides both.
bool dynamic_sched_from_env(bool by_default) {
  const char* v = std::getenv("BWG_SCHED");
  if (v == nullptr) return by_default;
  if (std::strcmp(v, "clc") == 0) return true;
  if (std::strcmp(v, "static") == 0) return false;
  return by_default;
}

int no_tail_split_from_env() {
  const char* v = std::getenv("BWG_NO_TAIL_SPLIT");
  return (v != nullptr && v[0] == '1') ? 1 : 0;
}

// Cluster split of the small-M kernel for few tiles: the cluster size F (2..8)
// that keeps the most SMs streaming, with every cluster co-resident
// (T <= clusters[F]) and at least two k-blocks per CTA; 1 if none helps.
// clusters == nullptr: a host-side estimate (76, 36 and 15 co-resident
// clusters of 2, 4 and 8 on 152 SMs, scaled to sm_count).
int small_m_split(int T, int kb, int sm_count, const int* clusters) {
  if (2 * T > sm_count) return 1;
  int best = 1;
  long long best_ctas = T;
  for (int f = 2; f <= kMaxSplit; ++f) {
    int c = 0;
    if (clusters != nullptr)
      c = clusters[f];
    else if (f == 2 || f == 4 || f == 8)
      c = (f == 2 ? sm_count / 2 : f == 4 ? sm_count * 36 / 152 : sm_count * 15 / 152);
    if (c < T || kb < 2 * f) continue;
    if (static_cast<long long>(T) * f > best_ctas) {
      best_ctas = static_cast<long long>(T) * f;
      best = f;
    }
  }
  return best;
}

bwg_status plan_dense(int M, int N, int K, int out_dtype, bool fp16_in, int sm_count, int max_smem,
                      int force_kernel, int force_stages, int max_clusters_2cta, int max_ctas_1cta,
                      int max_clusters_mc, int max_clusters_2c, bwg_plan_info* o,
                      const int* small_clusters = nullptr, bool force_streamk = false,
                      bool b_kmajor = false) {
  std::memset(o, 0, sizeof(*o));
  if (M == 0 || N == 0) {
    o->kernel = BWG_KERNEL_NONE;
    return BWG_OK;
  }
  if (K == 0) {
    o->kernel = BWG_KERNEL_ZERO;
    return BWG_OK;
  }
  int kind = force_kernel;
  if (kind == 0) {
    // 512x256 tiles (two MMA consumers per pair) do twice the MMA work of
    // 256x256 ones for each ring stage filled, and the filling of stages, not
    // the tensor pipe, is what limits the one-consumer tiles; use them while
    // they still give every pair at least one tile.
    const int pairs = max_clusters_2c > 0 ? max_clusters_2c : sm_count / 2;
    const long long tiles_2c = static_cast<long long>(ceil_div(M, 4 * kRowsPerCta)) * ceil_div(N, kTileN);
    if (M <= kSmallMMaxM)
      kind = BWG_KERNEL_SMALL_M;
    else if (tiles_2c >= pairs)
      kind = BWG_KERNEL_2CTA_2C;
    else
      kind = BWG_KERNEL_2CTA;
  }
  if (kind != BWG_KERNEL_1CTA && kind != BWG_KERNEL_2CTA && kind != BWG_KERNEL_SMALL_M &&
      kind != BWG_KERNEL_2CTA_MC && kind != BWG_KERNEL_2CTA_2C)
    return BWG_ERR_INVALID_ARG;
  if (kind == BWG_KERNEL_SMALL_M && M > kSmallMMaxM) return BWG_ERR_UNSUPPORTED;
  const uint32_t fmt = fp16_in ? kFmtF16 : kFmtBF16;
  o->kernel = kind;
  o->tile_k = kBK;
  o->k_blocks = ceil_div(K, kBK);
  if (kind == BWG_KERNEL_SMALL_M) {
    const int m_pad = small_m_pad(M);
    o->tile_m = m_pad;
    o->tile_n = 128;
    o->mma_m = 128;
    o->mma_n = m_pad;
    // 128 columns per tile by default: narrower strides start B's boxes off a
    // 128-byte boundary, which measured slower than leaving SMs idle.
    int tn = 128;
    const char* tn_env = force_streamk ? nullptr : std::getenv("BWG_SMALL_M_TILE_N");
    if (const char* v = tn_env) {
      const int f = std::atoi(v);
      if (f >= 16 && f <= 128 && f % 16 == 0) tn = f;
    }
    o->tile_n = tn;
    o->tiles = ceil_div(N, tn);
    const long long iters = static_cast<long long>(o->tiles) * o->k_blocks;
    // With at most half the SMs' worth of tiles, a cluster split of K keeps
    // more SMs streaming and sums the partials on chip (BWG_SMALL_M_SPLIT=0
    // turns it off, =F forces cluster size F where it is valid; BWG_STREAMK=1
    // takes stream-K instead).
    int split = o->tile_n == 128 ? small_m_split(o->tiles, o->k_blocks, sm_count, small_clusters) : 1;
    if (const char* v = std::getenv("BWG_SMALL_M_SPLIT")) {
      const int f = std::atoi(v);
      split = (f >= 2 && f <= kMaxSplit && o->tile_n == 128 && o->k_blocks >= 2 * f) ? f : 1;
    }
    // Stream-K pays when whole tiles would need a partly filled second wave,
    // or fill at most half the SMs; in between, whole tiles walking K in step
    // measured faster.
    int streamk = (o->tiles % sm_count != 0 && (o->tiles > sm_count || 2 * o->tiles <= sm_count) &&
                   iters >= sm_count && split == 1) ? 1 : 0;
    if (const char* v = std::getenv("BWG_STREAMK")) {
      streamk = (v[0] == '1' && iters >= sm_count) ? 1 : 0;
      if (streamk) split = 1;
    }
    if (force_streamk) {  // the no-allocation entry point: always stream-K
      streamk = 1;
      split = 1;
    }
    // With one tile per CTA the stage ring is idle when the epilogue runs, so
    // the output staging tile lives in it and the ring gets one stage deeper.
    const bool in_ring = !streamk && (split > 1 || o->tiles <= sm_count);
    const int fixed = small_m_smem(m_pad, out_dtype, 0, in_ring);
    int stages = std::min(8, (max_smem - fixed) / small_m_stage_bytes(m_pad));
    if (force_stages > 0) stages = force_stages;
    if (stages < 2 || small_m_smem(m_pad, out_dtype, stages, in_ring) > max_smem) return BWG_ERR_UNSUPPORTED;
    o->stages = stages;
    o->smem_input_per_cta = stages * small_m_stage_bytes(m_pad);
    o->smem_total = small_m_smem(m_pad, out_dtype, stages, in_ring);
    o->staging_in_ring = in_ring ? 1 : 0;
    o->bt_loads = small_m_one_bt_box(N, o->tile_n, b_kmajor) ? 1 : 2;
    o->pair_loads = small_m_pairs_ok(N, K, o->tile_n, stages, b_kmajor) ? 1 : 0;
    // each CTA's partial and the rows it receives fit in its idle stage ring
    if (split > 1 && (static_cast<long long>(m_pad) + static_cast<long long>(split) * ceil_div(M, split)) * 512 >
                         static_cast<long long>(stages) * small_m_stage_bytes(m_pad))
      split = 1;
    o->streamk = streamk;
    o->split = split;
    o->grid = streamk ? sm_count : split > 1 ? o->tiles * split : std::min(o->tiles, sm_count);
    o->tx_bytes = static_cast<uint32_t>(small_m_stage_bytes(m_pad));
    o->idesc = make_idesc_f16(fmt, /*a_mn_major=*/!b_kmajor, /*b_mn_major=*/false, 128, m_pad);
  } else {
    const int cg = (kind == BWG_KERNEL_1CTA) ? 1 : 2;
    const int mc = (kind == BWG_KERNEL_2CTA_MC) ? 2 : 1;  // pairs per cluster
    const int nc = (kind == BWG_KERNEL_2CTA_2C) ? 2 : 1;  // MMA consumers per pair
    const bool direct = direct_store_from_env();
    o->tile_m = kRowsPerCta * cg * nc;
    o->tile_n = kTileN;
    o->mma_m = kRowsPerCta * cg;
    o->mma_n = kTileN;
    const int fixed = dense_smem(cg, 0, direct, nc);
    int stages = std::min(8, (max_smem - fixed) / dense_stage_bytes(cg, nc));
    if (force_stages > 0) stages = force_stages;
    if (stages < 2 || dense_smem(cg, stages, direct, nc) > max_smem) return BWG_ERR_UNSUPPORTED;
    o->stages = stages;
    o->tiles = ceil_div(M, o->tile_m) * ceil_div(N, o->tile_n);
    o->smem_input_per_cta = stages * dense_stage_bytes(cg, nc);
    o->smem_total = dense_smem(cg, stages, direct, nc);
    if (nc == 2) {
      o->workers = std::min(o->tiles, max_clusters_2c > 0 ? max_clusters_2c : sm_count / 2);
      o->grid = 2 * o->workers;
    } else if (mc == 2) {
      // schedule units are stacks of two pair tiles; 4-CTA clusters
      const int units = ceil_div(ceil_div(M, o->tile_m), 2) * ceil_div(N, o->tile_n);
      o->workers = std::min(units, max_clusters_mc > 0 ? max_clusters_mc : sm_count / 4);
      o->grid = 4 * o->workers;
    } else if (cg == 2) {
      o->workers = std::min(o->tiles, max_clusters_2cta > 0 ? max_clusters_2cta : sm_count / 2);
      o->grid = 2 * o->workers;
    } else {
      o->workers = std::min(o->tiles, max_ctas_1cta > 0 ? max_ctas_1cta : sm_count);
      o->grid = o->workers;
    }
    o->tx_bytes = static_cast<uint32_t>(cg * dense_stage_bytes(cg, nc));
    o->idesc = make_idesc_f16(fmt, /*a_mn_major=*/false, /*b_mn_major=*/!b_kmajor, o->mma_m, kTileN);
  }
  o->coverage = static_cast<double>(M) * N / (static_cast<double>(o->tiles) * o->tile_m * o->tile_n);
  o->units = o->tiles;
  if (kind != BWG_KERNEL_SMALL_M) {
    const int per_unit = kind == BWG_KERNEL_2CTA_MC ? 2 : 1;
    const int base_units = ceil_div(ceil_div(M, o->tile_m), per_unit) * ceil_div(N, o->tile_n);
    int f = 1;
    const bool two = kind == BWG_KERNEL_2CTA_2C;
    const int R = no_tail_split_from_env()
                      ? 0
                      : tail_split(base_units, o->workers, two ? 4 : 2, two ? kCostHalf2 : kCostHalf1,
                                   kCostQuarter2, &f);
    o->units = base_units - R + R * f;
    if (two && dynamic_sched_from_env(false)) {
      o->dynamic = 1;
      o->grid = 2 * o->units;  // one pair per unit; running pairs claim the rest
    } else if (two) {
      // stream-K last wave, if it beats the (cut or uncut) last wave; it
      // spreads over every pair that fits, also when there are fewer tiles
      const int C = max_clusters_2c > 0 ? max_clusters_2c : sm_count / 2;
      const int cut_cost =
          R == 0 ? 1000 : ceil_div(f * R, o->workers) * (f == 2 ? kCostHalf2 : kCostQuarter2);
      // Opt-in (BWG_STREAMK_DENSE=1 takes it whenever it applies): measured
      // on GB300 it does not pay.  Pairs working at unrelated k offsets of
      // different tiles share no A or B data in L2, so the stream-K phase is
      // DRAM-bound at about 1.6x the per-k-block time of the lock-stepped
      // whole-tile waves, which cancels the better balance (4096^3: 94.8 vs
      // 92.8 us; 4096^2 x 16384: 339 vs 308 us).
      const char* env = std::getenv("BWG_STREAMK_DENSE");
      int segs = 0;
      int sk = 0;
      if (env != nullptr && env[0] == '1')
        sk = streamk_tiles(base_units, C, o->k_blocks, 1 << 30, &segs);
      (void)cut_cost;
      if (sk > 0) {
        o->streamk = 1;
        o->sk_tiles = sk;
        o->sk_segs = segs;
        o->workers = C;
        o->grid = 2 * C;
        o->units = segs * C + base_units - sk;
      }
    }
  } else {
    o->workers = o->grid;
  }
  return BWG_OK;
}

int out_elt(int out_dtype) { return out_dtype == BWG_OUT_FP32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// b_kmajor: B is stored [N, K] (ldb >= K) instead of [K, N] (ldb >= N).
bwg_status check_args(const void* A, const void* B, const void* D, int M, int N, int K, int lda,
                      int ldb, int ldd, int out_dtype, bool b_kmajor = false) {
  if (out_dtype != BWG_OUT_BF16 && out_dtype != BWG_OUT_FP32 && out_dtype != BWG_OUT_FP16)
    return BWG_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return BWG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return BWG_OK;
  if (D == nullptr || ldd < N) return BWG_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < (b_kmajor ? K : N)))
    return BWG_ERR_INVALID_ARG;
  if (!aligned16(D) || (static_cast<long long>(ldd) * out_elt(out_dtype)) % 16 != 0)
    return BWG_ERR_ALIGNMENT;
  if (K > 0 && (!aligned16(A) || !aligned16(B) || (static_cast<long long>(lda) * 2) % 16 != 0 ||
                (static_cast<long long>(ldb) * 2) % 16 != 0))
    return BWG_ERR_ALIGNMENT;
  return BWG_OK;
}

// ------------------------------------------------------------- devices -----

bwg_status ensure_device(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BWG_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return BWG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    st.ready = true;
    st.init_status = BWG_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&st.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      st.init_status = BWG_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      st.init_status = BWG_ERR_UNSUPPORTED;  // the library carries sm_103a code only
    }
    if (st.init_status == BWG_OK && g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        st.init_status = BWG_ERR_CUDA;
      } else {
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    if (st.init_status == BWG_OK) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess ||
          cudaMemset(p, 0, sizeof(unsigned long long)) != cudaSuccess) {
        cudaGetLastError();
        st.init_status = BWG_ERR_CUDA;
      } else {
        st.err = static_cast<unsigned long long*>(p);
      }
    }
    if (st.init_status == BWG_OK) {
      if (set_gemm_attributes(st.max_smem) != cudaSuccess ||
          set_small_m_attributes(st.max_smem) != cudaSuccess) {
        cudaGetLastError();
        st.init_status = BWG_ERR_CUDA;
      } else {
        st.clusters_2cta = max_active_clusters_gemm(2, false, dense_smem(2, 6));
        st.clusters_mc = max_active_clusters_gemm(4, false, dense_smem(2, 6));
        st.clusters_2c = max_active_clusters_gemm_2c(dense_smem(2, 4, false, 2));
        st.clusters_grouped_2c = max_active_clusters_grouped_2c(dense_smem(2, 4, false, 2));
        st.clusters_grouped = max_active_clusters_gemm(2, true, dense_smem(2, 6));
        st.ctas_1cta = max_active_clusters_gemm(1, false, dense_smem(1, 4));
        if (st.clusters_2cta <= 0) st.clusters_2cta = st.sm_count / 2;
        if (st.clusters_mc <= 0) st.clusters_mc = st.sm_count / 4;
        if (st.clusters_2c <= 0) st.clusters_2c = st.sm_count / 2;
        if (st.clusters_grouped_2c <= 0) st.clusters_grouped_2c = st.sm_count / 2;
        if (st.clusters_grouped <= 0) st.clusters_grouped = st.sm_count / 2;
        if (st.ctas_1cta <= 0) st.ctas_1cta = st.sm_count;
        // every small-M configuration takes more than half an SM's shared
        // memory, so one query at the largest size holds for all of them
        for (int f = 2; f <= kMaxSplit; ++f)
          st.clusters_small[f] = max_active_clusters_small_m(f, static_cast<size_t>(st.max_smem));
      }
    }
  }
  *out = &st;
  return st.init_status;
}

// Tensor map of a rank-`rank` view (2 to 4 dimensions, innermost first;
// strides in bytes for dimensions 1.., box in elements), cached by its
// arguments.
bool get_map_nd(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, int rank,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                CUtensorMapSwizzle swizzle) {
  int dev = 0;
  cudaGetDevice(&dev);
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.ptr = ptr;
  for (int d = 0; d < rank; ++d) {
    key.dims[d] = dims[d];
    key.box[d] = box[d];
    if (d + 1 < rank) key.strides[d] = strides[d];
  }
  key.rank = rank;
  key.dtype = static_cast<int>(dtype);
  key.swizzle = static_cast<int>(swizzle);
  key.device = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_maps.find(key);
  if (it != g_maps.end()) {
    *m = it->second;
    return true;
  }
  cuuint64_t gdim[4], gstride[3];
  cuuint32_t bx[4], estride[4] = {1, 1, 1, 1};
  for (int d = 0; d < rank; ++d) {
    gdim[d] = dims[d];
    bx[d] = box[d];
    if (d + 1 < rank) gstride[d] = strides[d];
  }
  CUtensorMap map;
  if (g_encode(&map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), gdim, gstride, bx,
               estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (g_maps.size() > 8192) g_maps.clear();
  g_maps.emplace(key, map);
  *m = map;
  return true;
}

// 2-D map of a row-major matrix: `inner` elements per row, `outer` rows,
// `row_bytes` apart.
bool get_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
             uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {inner, outer};
  const uint32_t box[2] = {box_inner, box_outer};
  return get_map_nd(m, ptr, dtype, 2, dims, &row_bytes, box, swizzle);
}

// B^T maps of the small-M kernel (single stage and, where the layout
// allows, two stages per load) and the two-stage map of A; sets bt_boxes and
// pair_loads.  Row-major B with N or the tile stride not a multiple of 64 is
// loaded as two 64-channel boxes a stage.
bool small_m_operand_maps(SmallMParams* p, const void* A, const void* B, CUtensorMapDataType in_t,
                          int M, int N, int K, long long lda, long long ldb, int m_pad, int tile_n,
                          int stages, bool b_kmajor) {
  const uint64_t bs = static_cast<uint64_t>(ldb) * 2;
  const uint64_t as = static_cast<uint64_t>(lda) * 2;
  const bool pairs = small_m_pairs_ok(N, K, tile_n, stages, b_kmajor);
  if (b_kmajor) {
    // B [N, K]: one box of 128 rows (channels) x 64 K a stage
    if (!get_map(&p->map_bt, B, in_t, K, N, bs, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    p->bt_boxes = 1;
  } else if (small_m_one_bt_box(N, tile_n, false)) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64)};
    const uint64_t strides[2] = {bs, 128};
    const uint32_t box[3] = {64, 64, 2};
    if (!get_map_nd(&p->map_bt, B, in_t, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    p->bt_boxes = 1;
  } else {
    if (!get_map(&p->map_bt, B, in_t, N, K, bs, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    p->bt_boxes = 2;
  }
  p->pair_loads = 0;
  if (!pairs) return true;
  const uint64_t kb = static_cast<uint64_t>(K / 64);
  if (b_kmajor) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(N), kb};
    const uint64_t strides[2] = {bs, 128};
    const uint32_t box[3] = {64, 128, 2};
    if (!get_map_nd(&p->map_bt2, B, in_t, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  } else {
    const uint64_t dims[4] = {64, 64, static_cast<uint64_t>(N / 64), kb};
    const uint64_t strides[3] = {bs, 128, 64 * bs};
    const uint32_t box[4] = {64, 64, 2, 2};
    if (!get_map_nd(&p->map_bt2, B, in_t, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  }
  const uint64_t adims[3] = {64, static_cast<uint64_t>(M), kb};
  const uint64_t astrides[2] = {as, 128};
  const uint32_t abox[3] = {64, static_cast<uint32_t>(m_pad), 2};
  if (!get_map_nd(&p->map_at2, A, in_t, 3, adims, astrides, abox, CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  p->pair_loads = 1;
  return true;
}

int force_kernel_from_env() {
  const char* v = std::getenv("BWG_FORCE_KERNEL");
  if (v == nullptr) return 0;
  if (!std::strcmp(v, "1cta")) return BWG_KERNEL_1CTA;
  if (!std::strcmp(v, "2cta")) return BWG_KERNEL_2CTA;
  if (!std::strcmp(v, "2cta_mc")) return BWG_KERNEL_2CTA_MC;
  if (!std::strcmp(v, "2cta_2c")) return BWG_KERNEL_2CTA_2C;
  if (!std::strcmp(v, "small_m")) return BWG_KERNEL_SMALL_M;
  return 0;
}

int force_stages_from_env() {
  const char* v = std::getenv("BWG_FORCE_STAGES");
  return v ? std::atoi(v) : 0;
}

CUtensorMapDataType out_map_dtype(int out_dtype) {
  if (out_dtype == BWG_OUT_FP32) return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (out_dtype == BWG_OUT_FP16) return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// Whether p points into device memory of the current device (allocated on
// it with cudaMalloc or a pool on it).
bool local_device_memory(const void* p) {
  int dev = 0;
  cudaPointerAttributes a;
  std::memset(&a, 0, sizeof(a));
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

bwg_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return BWG_OK;
  cudaGetLastError();
  return BWG_ERR_CUDA;
}

bwg_status run_dense(bool fp16_in, const void* A, const void* B, void* D, int M, int N, int K,
                     int lda, int ldb, int ldd, int out_dtype, cudaStream_t stream,
                     bool b_kmajor = false) {
  bwg_status s = check_args(A, B, D, M, N, K, lda, ldb, ldd, out_dtype, b_kmajor);
  if (s != BWG_OK) return s;
  if (M == 0 || N == 0) return BWG_OK;
  DeviceState* st = nullptr;
  if ((s = ensure_device(&st)) != BWG_OK) return s;
  bwg_plan_info pl;
  s = plan_dense(M, N, K, out_dtype, fp16_in, st->sm_count, st->max_smem, force_kernel_from_env(),
                 force_stages_from_env(), st->clusters_2cta, st->ctas_1cta, st->clusters_mc,
                 st->clusters_2c, &pl, st->clusters_small, false, b_kmajor);
  if (s != BWG_OK) return s;
  if (pl.kernel == BWG_KERNEL_ZERO)
    return launch_status(launch_zero_fill(D, M, N, ldd, out_elt(out_dtype), stream));
  const CUtensorMapDataType in_t =
      fp16_in ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int oe = out_elt(out_dtype);
  if (pl.kernel == BWG_KERNEL_SMALL_M) {
    SmallMParams p;
    std::memset(&p, 0, sizeof(p));
    const int m_pad = pl.mma_n;
    if (!small_m_operand_maps(&p, A, B, in_t, M, N, K, lda, ldb, m_pad, pl.tile_n, pl.stages,
                              b_kmajor) ||
        !get_map(&p.map_at, A, in_t, K, M, static_cast<uint64_t>(lda) * 2, kBK, m_pad,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
        !get_map(&p.map_d, D, out_map_dtype(out_dtype), N, M, static_cast<uint64_t>(ldd) * oe,
                 std::min(64, pl.tile_n), m_pad, CU_TENSOR_MAP_SWIZZLE_NONE))
      return BWG_ERR_CUDA;
    if (pl.tile_n > 64 &&
        !get_map(&p.map_d2, D, out_map_dtype(out_dtype), N, M, static_cast<uint64_t>(ldd) * oe,
                 pl.tile_n - 64, m_pad, CU_TENSOR_MAP_SWIZZLE_NONE))
      return BWG_ERR_CUDA;
    p.tile_n = pl.tile_n;
    p.err = st->err;
    p.timeout_ns = g_timeout_ns.load();
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_pad = m_pad;
    p.num_tiles = pl.tiles;
    p.num_k_blocks = pl.k_blocks;
    p.stages = pl.stages;
    p.out_dtype = out_dtype;
    p.idesc = pl.idesc;
    p.tx_extra = g_tx_extra.load();
    p.streamk = pl.streamk;
    p.split = pl.split;
    p.b_kmajor = b_kmajor ? 1 : 0;
    p.staging_in_ring = pl.staging_in_ring;
    // B^T streams through L2 as evict-first (whole tiles and stream-K; the
    // cluster split measured 5% slower with it); BWG_SMALL_M_L2HINT
    // overrides (bit 1: B^T evict-first, bit 0: A evict-last).
    p.l2hint = pl.split > 1 ? 0 : 2;
    if (const char* v = std::getenv("BWG_SMALL_M_L2HINT")) p.l2hint = std::atoi(v) & 3;
    p.d = D;
    p.ldd = ldd;
    p.trace = g_trace.load();
    if (pl.streamk) {
      p.ws_slots = streamk_max_sharers(pl.tiles, pl.k_blocks, pl.grid);
      Workspace w;
      const size_t ws_bytes = static_cast<size_t>(pl.tiles) * p.ws_slots * m_pad * 128 * sizeof(float);
      if ((s = get_workspace(stream, ws_bytes, pl.tiles, &w)) != BWG_OK) return s;
      p.ws = w.ws;
      p.ws_counters = w.counters;
    }
    return launch_status(launch_small_m(p, pl.grid, pl.smem_total, stream));
  }
  // The multicast kernel's loads land in the shared memory of two CTA pairs
  // at once; it may read only memory that this GPU owns.  Anything else (host
  // memory, another GPU's memory, managed memory) is refused before any
  // descriptor is made or any kernel launched.
  if (pl.kernel == BWG_KERNEL_2CTA_MC &&
      (!local_device_memory(A) || !local_device_memory(B)))
    return BWG_ERR_INVALID_ARG;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  const uint32_t d_box_inner = out_dtype == BWG_OUT_FP32 ? 32 : 64;
  if (!get_map(&p.map_a, A, in_t, K, M, static_cast<uint64_t>(lda) * 2, kBK, kRowsPerCta,
               CU_TENSOR_MAP_SWIZZLE_128B) ||
      !get_map(&p.map_b, B, in_t, b_kmajor ? K : N, b_kmajor ? N : K, static_cast<uint64_t>(ldb) * 2,
               64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !get_map(&p.map_d, D, out_map_dtype(out_dtype), N, M, static_cast<uint64_t>(ldd) * oe,
               d_box_inner, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return BWG_ERR_CUDA;
  {
    // One B load a stage per pair CTA (its two 64-column chunks): [K, N] as
    // a 3-D view, which needs N a multiple of 64 so that no chunk reaches past
    // a row; [N, K] as a 128-row box.  BWG_B_ONE_BOX=0 turns it off.
    const char* v = std::getenv("BWG_B_ONE_BOX");
    const bool on = !(v != nullptr && v[0] == '0') && (b_kmajor || N % 64 == 0);
    if (on) {
      bool ok;
      if (b_kmajor) {
        ok = get_map(&p.map_b1, B, in_t, K, N, static_cast<uint64_t>(ldb) * 2, 64, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B);
      } else {
        const uint64_t dims[3] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64)};
        const uint64_t strides[2] = {static_cast<uint64_t>(ldb) * 2, 128};
        const uint32_t box[3] = {64, 64, 2};
        ok = get_map_nd(&p.map_b1, B, in_t, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      }
      if (!ok) return BWG_ERR_CUDA;
      p.b_one_box = 1;
    }
  }
  p.err = st->err;
  p.d_ptr = D;
  p.timeout_ns = g_timeout_ns.load();
  p.M = M;
  p.N = N;
  p.K = K;
  p.ldd = ldd;
  p.b_kmajor = b_kmajor ? 1 : 0;
  p.num_m_tiles = ceil_div(M, pl.tile_m);
  p.num_n_tiles = ceil_div(N, pl.tile_n);
  p.num_k_blocks = pl.k_blocks;
  p.group_m = group_m_from_env();
  p.stages = pl.stages;
  p.out_dtype = out_dtype;
  p.idesc = pl.idesc;
  p.tx_extra = g_tx_extra.load();
  p.trace = g_trace.load();
  p.no_tail_split = no_tail_split_from_env();
  p.direct_store = direct_store_from_env() ? 1 : 0;
  if (pl.kernel == BWG_KERNEL_2CTA)
    return launch_status(launch_gemm_2cta(p, pl.grid, pl.smem_total, stream));
  if (pl.kernel == BWG_KERNEL_2CTA_MC)
    return launch_status(launch_gemm_2cta_mc(p, pl.grid, pl.smem_total, stream));
  p.workers = pl.workers;
  if (pl.kernel == BWG_KERNEL_2CTA_2C && pl.streamk) {
    p.sk_tiles = pl.sk_tiles;
    p.sk_segs = pl.sk_segs;
    p.ws_slots = streamk_max_sharers(pl.sk_tiles, pl.k_blocks, pl.workers);
    const size_t ws_bytes = static_cast<size_t>(pl.sk_tiles) * p.ws_slots * 16u * 32u * kTileN * 4u;
    Workspace w;
    bwg_status ws = get_workspace(stream, ws_bytes, pl.sk_tiles * 16, &w);
    if (ws != BWG_OK) return ws;
    p.ws = w.ws;
    p.ws_counters = w.counters;
  }
  if (pl.kernel == BWG_KERNEL_2CTA_2C)
    return launch_status(launch_gemm_2cta_2c(p, pl.grid, pl.smem_total, stream, pl.dynamic != 0));
  return launch_status(launch_gemm_1cta(p, pl.grid, pl.smem_total, stream));
}

// swiglu: B_g is [gate | up] with N columns (N/2 each) and D is H [M_total,
// N/2] = silu(gate) * up.  The up block starts at column N/2, which a TMA
// load's first coordinate must reach on a 16-byte boundary: N/2 a multiple
// of 8, i.e. N a multiple of 16.
// b_kmajor: each B[g] is stored [N, K] (the pages' layout) instead of [K, N].
bwg_status run_grouped(bool fp16, const void* A, const void* const* B, void* D,
                       const int* group_offsets, int G, int M_total, int N, int K,
                       cudaStream_t stream, bool swiglu = false, bool b_kmajor = false) {
  if (G < 0 || M_total < 0 || N < 0 || K < 0) return BWG_ERR_INVALID_ARG;
  if (G == 0 || M_total == 0 || N == 0) return BWG_OK;
  if (D == nullptr || group_offsets == nullptr) return BWG_ERR_INVALID_ARG;
  if (!aligned16(D) || (static_cast<long long>(N) * 2) % 16 != 0) return BWG_ERR_ALIGNMENT;
  if (swiglu && N % 16 != 0) return BWG_ERR_ALIGNMENT;
  const int n_out = swiglu ? N / 2 : N;  // columns of D
  if (K > 0) {
    if (A == nullptr || B == nullptr) return BWG_ERR_INVALID_ARG;
    if (!aligned16(A) || (static_cast<long long>(K) * 2) % 16 != 0) return BWG_ERR_ALIGNMENT;
    for (int g = 0; g < G; ++g) {
      if (B[g] == nullptr) return BWG_ERR_INVALID_ARG;
      if (!aligned16(B[g])) return BWG_ERR_ALIGNMENT;
    }
  }
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  // K = 0: every accumulator is 0, and so is silu(0) * 0
  if (K == 0) return launch_status(launch_zero_fill(D, M_total, n_out, n_out, 2, stream));
  const CUtensorMapDataType in_t =
      fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // Two MMA consumers (512-row units) unless BWG_GROUPED_1C=1 asks for the
  // 256-row kernel; the one-consumer kernel is also the one with swapped ends.
  const char* one_env = std::getenv("BWG_GROUPED_1C");
  const bool two = !(one_env != nullptr && one_env[0] == '1');
  const int nc = two ? 2 : 1;
  const int stages = force_stages_from_env() > 0 ? force_stages_from_env() : (two ? 4 : 6);
  const int smem = dense_smem(2, stages, false, nc);
  if (smem > st->max_smem) return BWG_ERR_UNSUPPORTED;
  for (int g0 = 0; g0 < G; g0 += kMaxGroupsPerLaunch) {
    const int gn = std::min(kMaxGroupsPerLaunch, G - g0);
    GroupedParams P;
    std::memset(&P, 0, sizeof(P));
    GemmParams& p = P.base;
    if (!get_map(&p.map_a, A, in_t, K, M_total, static_cast<uint64_t>(K) * 2, kBK, kRowsPerCta,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
        !get_map(&p.map_d, D, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 n_out, M_total, static_cast<uint64_t>(n_out) * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
      return BWG_ERR_CUDA;
    for (int i = 0; i < gn; ++i)
      if (!get_map(&P.map_b[i], B[g0 + i], in_t, b_kmajor ? K : N, b_kmajor ? N : K,
                   static_cast<uint64_t>(b_kmajor ? K : N) * 2, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return BWG_ERR_CUDA;
    p.err = st->err;
    p.d_ptr = D;
    p.group_offsets = group_offsets;
    p.timeout_ns = g_timeout_ns.load();
    p.M = M_total;
    p.N = n_out;
    p.K = K;
    p.ldd = n_out;
    p.num_n_tiles = ceil_div(n_out, swiglu ? kTileN / 2 : kTileN);
    p.swiglu_up = swiglu ? n_out : 0;
    p.num_m_tiles = 0;
    p.num_k_blocks = ceil_div(K, kBK);
    p.group_m = kGroupM;
    p.stages = stages;
    p.out_dtype = fp16 ? BWG_OUT_FP16 : BWG_OUT_BF16;
    p.idesc = make_idesc_f16(fp16 ? kFmtF16 : kFmtBF16, false, !b_kmajor, 2 * kRowsPerCta, kTileN);
    p.b_kmajor = b_kmajor ? 1 : 0;
    p.tx_extra = g_tx_extra.load();
    p.trace = g_trace.load();
    p.G = gn;
    p.g_begin = g0;
    p.G_total = G;
    p.no_tail_split = no_tail_split_from_env();
    p.idesc_swap = make_idesc_f16(fp16 ? kFmtF16 : kFmtBF16, true, false, 2 * kRowsPerCta, 16);
    {
      // Off by default: a swapped tile still loads whole A and B boxes, and
      // tiles here are bound by how fast shared memory fills, so it measured
      // no faster than the padded tile.  BWG_GROUPED_SWAP=1 turns it on.
      const char* v = std::getenv("BWG_GROUPED_SWAP");
      p.swap_ends = (v != nullptr && v[0] == '1' && !swiglu && !b_kmajor) ? 1 : 0;
    }
    // Upper bound on tiles: every group adds at most one partial row tile.
    const long long max_tiles =
        (static_cast<long long>(ceil_div(M_total, 2 * kRowsPerCta * nc)) + gn) * p.num_n_tiles;
    const int clusters = static_cast<int>(
        std::min<long long>(max_tiles, two ? st->clusters_grouped_2c : st->clusters_grouped));
    // Dynamic scheduling: one pair per unit.  The tile count is known only on
    // the device; the units of a last wave cut in up to 4 parts are at most
    // tiles + 3 x (pairs running at once), and pairs past the end claim or
    // find nothing.
    const bool dyn = two && dynamic_sched_from_env(true);
    p.workers = clusters;
    const long long grid_pairs = dyn ? max_tiles + 3LL * clusters : clusters;
    if (2 * grid_pairs > 0x7fffffffLL) return BWG_ERR_UNSUPPORTED;
    const cudaError_t e =
        two ? launch_grouped_2c(P, static_cast<int>(2 * grid_pairs), smem, stream, swiglu, dyn)
            : launch_grouped_2cta(P, 2 * clusters, smem, stream, swiglu);
    if (e != cudaSuccess) return launch_status(e);
  }
  return BWG_OK;
}

// ------------------------------------------- no-allocation small-M path -----
//
// Some callers cannot let a library call cudaMalloc: processes that hand all
// device memory to their own pool allocator up front (an allocation from the
// library would fail or eat into that budget), and real-time loops that must
// not block on the allocator (cudaMalloc can stall the host and synchronise
// the device).  For
// them gemm_bf16_small_m_noalloc runs the stream-K small-M kernel with its
// partial sums and tile counters in the fixed device array below instead of
// the per-stream workspace that gemm_bf16 allocates.
//
// The array is a plain global of the library: every GPU that loads the
// library holds these 32 MiB until the process exits, all calls on a device
// share them, and each call leaves its partial sums behind.  Calls whose GPU
// work overlaps (different streams, no ordering between them) race on it.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // whole array
constexpr size_t kNoAllocCounterBytes = size_t(64) << 10;   // tile counters: up to 16384 tiles
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array for the current device.  The name
// g_noalloc_scratch in host code is only a handle for the runtime, so the
// address is looked up once per device (with that device current) and kept.
bwg_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return launch_status(cudaErrorUnknown);
  if (dev < 0 || dev >= kMaxDevices) return BWG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return BWG_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return BWG_OK;
}

// Tensor map without the descriptor cache (inserting into the cache would
// allocate host memory).
bool encode_map_direct(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
                       uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                       CUtensorMapSwizzle swizzle) {
  cuuint64_t gdim[2] = {inner, outer};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estride[2] = {1, 1};
  return g_encode(m, dtype, 2, const_cast<void*>(ptr), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bwg_status run_small_m_noalloc(const void* A, const void* B, void* D, int M, int N, int K, int lda,
                               int ldb, int ldd, int out_dtype, cudaStream_t stream) {
  bwg_status s = check_args(A, B, D, M, N, K, lda, ldb, ldd, out_dtype);
  if (s != BWG_OK) return s;
  if (M == 0 || N == 0) return BWG_OK;
  if (M > kSmallMMaxM) return BWG_ERR_UNSUPPORTED;
  DeviceState* st = nullptr;
  if ((s = ensure_device(&st)) != BWG_OK) return s;
  if (K == 0) return launch_status(launch_zero_fill(D, M, N, ldd, out_elt(out_dtype), stream));
  bwg_plan_info pl;
  s = plan_dense(M, N, K, out_dtype, false, st->sm_count, st->max_smem, BWG_KERNEL_SMALL_M, 0,
                 st->clusters_2cta, st->ctas_1cta, st->clusters_mc, st->clusters_2c, &pl, nullptr, true);
  if (s != BWG_OK) return s;
  // Always the stream-K form: every CTA gets at least one k-block.
  const long long iters = static_cast<long long>(pl.tiles) * pl.k_blocks;
  const int grid = static_cast<int>(std::min<long long>(st->sm_count, iters));
  const int m_pad = pl.mma_n;
  const int slots = streamk_max_sharers(pl.tiles, pl.k_blocks, grid);
  const size_t counter_bytes = static_cast<size_t>(pl.tiles) * sizeof(int);
  const size_t partial_bytes = static_cast<size_t>(pl.tiles) * slots * m_pad * 128 * sizeof(float);
  if (counter_bytes > kNoAllocCounterBytes ||
      partial_bytes > kNoAllocScratchBytes - kNoAllocCounterBytes)
    return BWG_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != BWG_OK) return s;
  // The counters must start at zero; a call cut short by the watchdog could
  // have left some behind, so clear the ones this call uses.
  if (cudaMemsetAsync(scratch, 0, counter_bytes, stream) != cudaSuccess)
    return launch_status(cudaErrorUnknown);
  const CUtensorMapDataType in_t = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int oe = out_elt(out_dtype);
  SmallMParams p;
  std::memset(&p, 0, sizeof(p));
  p.bt_boxes = 2;  // two 2-D boxes a stage, one stage a load
  if (!encode_map_direct(&p.map_bt, B, in_t, N, K, static_cast<uint64_t>(ldb) * 2, 64, kBK,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_direct(&p.map_at, A, in_t, K, M, static_cast<uint64_t>(lda) * 2, kBK, m_pad,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_direct(&p.map_d, D, out_map_dtype(out_dtype), N, M,
                         static_cast<uint64_t>(ldd) * oe, 64, m_pad, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_map_direct(&p.map_d2, D, out_map_dtype(out_dtype), N, M,
                         static_cast<uint64_t>(ldd) * oe, 64, m_pad, CU_TENSOR_MAP_SWIZZLE_NONE))
    return BWG_ERR_CUDA;
  p.err = st->err;
  p.timeout_ns = g_timeout_ns.load();
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_pad = m_pad;
  p.tile_n = 128;
  p.num_tiles = pl.tiles;
  p.num_k_blocks = pl.k_blocks;
  p.stages = pl.stages;
  p.out_dtype = out_dtype;
  p.idesc = pl.idesc;
  p.tx_extra = g_tx_extra.load();
  p.streamk = 1;
  p.l2hint = 2;  // B^T evict-first, as in gemm_bf16
  p.ws_slots = slots;
  p.ws_counters = static_cast<int*>(scratch);
  p.ws = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kNoAllocCounterBytes);
  return launch_status(launch_small_m(p, grid, pl.smem_total, stream));
}

}  // namespace

// ================================================================ C ABI ====

extern "C" {

bwg_status gemm_bf16(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                     int ldd, int out_dtype, void* stream) {
  return run_dense(false, A, B, D, M, N, K, lda, ldb, ldd, out_dtype,
                   static_cast<cudaStream_t>(stream));
}

bwg_status gemm_fp16(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                     int ldd, int out_dtype, void* stream) {
  return run_dense(true, A, B, D, M, N, K, lda, ldb, ldd, out_dtype,
                   static_cast<cudaStream_t>(stream));
}

bwg_status grouped_gemm_bf16(const void* A, const void* const* B, void* D, const int* group_offsets,
                             int G, int M_total, int N, int K, void* stream) {
  return run_grouped(false, A, B, D, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream));
}

bwg_status grouped_gemm_fp16(const void* A, const void* const* B, void* D, const int* group_offsets,
                             int G, int M_total, int N, int K, void* stream) {
  return run_grouped(true, A, B, D, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream));
}

bwg_status grouped_gemm_swiglu_bf16(const void* A, const void* const* B, void* H,
                                    const int* group_offsets, int G, int M_total, int N, int K,
                                    void* stream) {
  return run_grouped(false, A, B, H, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), true);
}

bwg_status grouped_gemm_swiglu_fp16(const void* A, const void* const* B, void* H,
                                    const int* group_offsets, int G, int M_total, int N, int K,
                                    void* stream) {
  return run_grouped(true, A, B, H, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), true);
}

bwg_status gemm_bf16_nt(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                        int ldd, int out_dtype, void* stream) {
  return run_dense(false, A, B, D, M, N, K, lda, ldb, ldd, out_dtype,
                   static_cast<cudaStream_t>(stream), /*b_kmajor=*/true);
}

bwg_status gemm_fp16_nt(const void* A, const void* B, void* D, int M, int N, int K, int lda, int ldb,
                        int ldd, int out_dtype, void* stream) {
  return run_dense(true, A, B, D, M, N, K, lda, ldb, ldd, out_dtype,
                   static_cast<cudaStream_t>(stream), /*b_kmajor=*/true);
}

bwg_status grouped_gemm_bf16_nt(const void* A, const void* const* B, void* D,
                                const int* group_offsets, int G, int M_total, int N, int K,
                                void* stream) {
  return run_grouped(false, A, B, D, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), false, /*b_kmajor=*/true);
}

bwg_status grouped_gemm_fp16_nt(const void* A, const void* const* B, void* D,
                                const int* group_offsets, int G, int M_total, int N, int K,
                                void* stream) {
  return run_grouped(true, A, B, D, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), false, /*b_kmajor=*/true);
}

bwg_status grouped_gemm_swiglu_bf16_nt(const void* A, const void* const* B, void* H,
                                       const int* group_offsets, int G, int M_total, int N, int K,
                                       void* stream) {
  return run_grouped(false, A, B, H, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), true, /*b_kmajor=*/true);
}

bwg_status grouped_gemm_swiglu_fp16_nt(const void* A, const void* const* B, void* H,
                                       const int* group_offsets, int G, int M_total, int N, int K,
                                       void* stream) {
  return run_grouped(true, A, B, H, group_offsets, G, M_total, N, K,
                     static_cast<cudaStream_t>(stream), true, /*b_kmajor=*/true);
}

bwg_status gemm_bf16_small_m_noalloc(const void* A, const void* B, void* D, int M, int N, int K,
                                     int lda, int ldb, int ldd, int out_dtype, void* stream) {
  return run_small_m_noalloc(A, B, D, M, N, K, lda, ldb, ldd, out_dtype,
                             static_cast<cudaStream_t>(stream));
}

// Host-buffer product, pipelined over row chunks of A and D: B and the first
// chunk of A go up first; then chunk c's product runs on `stream` while chunk
// c+1 is copied in on one copy stream and chunk c-1's result goes back on the
// other, so the two copy directions and the tensor cores work at once.
bwg_status gemm_bf16_host(const void* A_host, const void* B_host, void* D_host, int M, int N, int K,
                          int out_dtype, void* dA, void* dB, void* dD, void* stream) {
  if (M < 0 || N < 0 || K < 0) return BWG_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (D_host == nullptr || (K > 0 && (A_host == nullptr || B_host == nullptr))))
    return BWG_ERR_INVALID_ARG;
  bwg_status s = check_args(dA, dB, dD, M, N, K, K, N, N, out_dtype);
  if (s != BWG_OK || M == 0 || N == 0) return s;
  DeviceState* st = nullptr;
  if ((s = ensure_device(&st)) != BWG_OK) return s;
  cudaStream_t us = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(st->host_mu);
  if (!st->host_ready) {
    bool ok = cudaStreamCreateWithFlags(&st->h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&st->d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&st->ev_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&st->ev_done, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < 8; ++c)
      ok = cudaEventCreateWithFlags(&st->ev_in[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&st->ev_out[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return launch_status(cudaErrorUnknown);
    st->host_ready = true;
  }
  // Chunks of whole 512-row tiles, at most 8, at least 1024 rows each.
  const int want = std::max(1, std::min(8, M / 1024));
  const int rows = ceil_div(ceil_div(M, want), 512) * 512;
  const int chunks = ceil_div(M, rows);
  const size_t oe = static_cast<size_t>(out_elt(out_dtype));
  auto a_at = [&](const void* base, int r) {
    return static_cast<const uint8_t*>(base) + static_cast<size_t>(r) * K * 2;
  };
  auto d_at = [&](void* base, int r) {
    return static_cast<uint8_t*>(base) + static_cast<size_t>(r) * N * oe;
  };
  auto fail = [&](cudaError_t e) { return e == cudaSuccess ? BWG_OK : launch_status(e); };
  // nothing starts before the work already on the caller's stream
  cudaError_t e = cudaEventRecord(st->ev_start, us);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st->h2d, st->ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st->d2h, st->ev_start, 0);
  if (e == cudaSuccess && K > 0)
    e = cudaMemcpyAsync(dB, B_host, static_cast<size_t>(K) * N * 2, cudaMemcpyHostToDevice, st->h2d);
  for (int c = 0; e == cudaSuccess && c < chunks; ++c) {
    const int r0 = c * rows, rc = std::min(rows, M - r0);
    if (K > 0)
      e = cudaMemcpyAsync(const_cast<uint8_t*>(a_at(dA, r0)), a_at(A_host, r0),
                          static_cast<size_t>(rc) * K * 2, cudaMemcpyHostToDevice, st->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(st->ev_in[c], st->h2d);
  }
  for (int c = 0; e == cudaSuccess && c < chunks; ++c) {
    const int r0 = c * rows, rc = std::min(rows, M - r0);
    e = cudaStreamWaitEvent(us, st->ev_in[c], 0);
    if (e != cudaSuccess) break;
    s = run_dense(false, a_at(dA, r0), dB, d_at(dD, r0), rc, N, K, K, N, N, out_dtype, us);
    if (s != BWG_OK) break;
    e = cudaEventRecord(st->ev_out[c], us);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st->d2h, st->ev_out[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(d_at(D_host, r0), d_at(dD, r0), static_cast<size_t>(rc) * N * oe,
                          cudaMemcpyDeviceToHost, st->d2h);
  }
  if (s != BWG_OK || e != cudaSuccess) {
    // Copies of this call may already be queued on the copy streams: let them
    // finish before returning, so that the caller may free or reuse its host
    // buffers as soon as it sees the error.
    cudaStreamSynchronize(st->h2d);
    cudaStreamSynchronize(st->d2h);
    cudaGetLastError();
    return s != BWG_OK ? s : fail(e);
  }
  // the caller's stream finishes after the last copy back
  e = cudaEventRecord(st->ev_done, st->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(us, st->ev_done, 0);
  return fail(e);
}

const char* bwg_status_string(int status) {
  switch (status) {
    case BWG_OK: return "ok";
    case BWG_ERR_INVALID_ARG: return "invalid argument";
    case BWG_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
    case BWG_ERR_UNSUPPORTED: return "unsupported device or size";
    case BWG_ERR_CUDA: return "CUDA runtime or driver error";
    case BWG_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case BWG_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the fixed 32 MiB no-allocation buffer holds";
    default: return "unknown status";
  }
}

bwg_status bwg_last_device_error(void* stream, unsigned long long* info) {
  if (info == nullptr) return BWG_ERR_INVALID_ARG;
  *info = 0;
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return launch_status(cudaErrorUnknown);
  unsigned long long w = 0;
  if (cudaMemcpy(&w, st->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(st->err, 0, sizeof(w)) != cudaSuccess)
    return launch_status(cudaErrorUnknown);
  *info = w;
  const unsigned long long kind = w >> 56;
  if (kind == kFaultTimeout) {
    // A kernel that gave up may have left stream-K arrival counters behind;
    // they must read zero at the start of every call.
    if (clear_workspace_counters() != BWG_OK) return BWG_ERR_CUDA;
    return BWG_ERR_TIMEOUT;
  }
  if (kind == kFaultBadOffsets) return BWG_ERR_INVALID_ARG;
  return BWG_OK;
}

bwg_status bwg_probe_cluster_pair(const float* in, float* sum_out, int* peer_out, int n,
                                  void* stream) {
  if (n <= 0 || (n & 1) || n > 65534 || in == nullptr || sum_out == nullptr || peer_out == nullptr)
    return BWG_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  return launch_status(
      launch_probe_cluster_pair(in, sum_out, peer_out, n, static_cast<cudaStream_t>(stream)));
}

bwg_status bwg_probe_tma_swizzle(const void* src, void* out, void* stream) {
  if (src == nullptr || out == nullptr) return BWG_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(out)) return BWG_ERR_ALIGNMENT;
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  CUtensorMap map;
  if (!encode_map_direct(&map, src, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, 64, 128, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return BWG_ERR_CUDA;
  return launch_status(launch_probe_tma_swizzle(map, out, st->err, g_timeout_ns.load(),
                                                static_cast<cudaStream_t>(stream)));
}

bwg_status bwg_probe_grouped_tables(const int* offsets, int g0, int G, int G_total, int M,
                                    int num_n_tiles, int tile_m, int* out, void* stream) {
  if (offsets == nullptr || out == nullptr || G < 1 || G > kMaxGroupsPerLaunch || g0 < 0 ||
      G_total < g0 + G || M < 0 || num_n_tiles < 1 || tile_m < 1)
    return BWG_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  return launch_status(launch_probe_grouped_tables(offsets, g0, G, G_total, M, num_n_tiles, tile_m, out,
                                                   static_cast<cudaStream_t>(stream)));
}

bwg_status bwg_probe_mma(const void* A, const void* B, float* D, int k_steps, int fp16,
                         void* stream) {
  if (A == nullptr || B == nullptr || D == nullptr || k_steps < 1 || k_steps > 4)
    return BWG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return BWG_ERR_ALIGNMENT;
  DeviceState* st = nullptr;
  bwg_status s = ensure_device(&st);
  if (s != BWG_OK) return s;
  const CUtensorMapDataType t = fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap ma, mb;
  if (!encode_map_direct(&ma, A, t, 64, 128, 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_map_direct(&mb, B, t, 256, 64, 512, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return BWG_ERR_CUDA;
  const uint32_t idesc = make_idesc_f16(fp16 ? kFmtF16 : kFmtBF16, false, true, 128, 256);
  return launch_status(launch_probe_mma(ma, mb, D, k_steps, idesc, st->err, g_timeout_ns.load(),
                                        static_cast<cudaStream_t>(stream)));
}

void bwg_set_watchdog_ns(unsigned long long ns) { g_timeout_ns.store(ns ? ns : 2000000000ull); }

void bwg_debug_set_tx_extra(unsigned int bytes) { g_tx_extra.store(bytes); }

void bwg_debug_set_trace(void* buffer) { g_trace.store(static_cast<unsigned long long*>(buffer)); }

bwg_status bwg_plan(int M, int N, int K, int out_dtype, int sm_count, int force_kernel,
                    int force_stages, bwg_plan_info* out) {
  if (out == nullptr || M < 0 || N < 0 || K < 0 || sm_count <= 0) return BWG_ERR_INVALID_ARG;
  if (out_dtype != BWG_OUT_BF16 && out_dtype != BWG_OUT_FP32 && out_dtype != BWG_OUT_FP16)
    return BWG_ERR_INVALID_ARG;
  // 227 KiB of opt-in shared memory per block on sm_100-family parts.
  return plan_dense(M, N, K, out_dtype, false, sm_count, 232448, force_kernel, force_stages, 0, 0, 0,
                    0, out);
}

bwg_status bwg_check_gemm_args(const void* A, const void* B, const void* D, int M, int N, int K,
                               int lda, int ldb, int ldd, int out_dtype) {
  return check_args(A, B, D, M, N, K, lda, ldb, ldd, out_dtype);
}

uint32_t bwg_idesc_f16(int bf16, int a_mn_major, int b_mn_major, int m, int n) {
  return make_idesc_f16(bf16 ? kFmtBF16 : kFmtF16, a_mn_major != 0, b_mn_major != 0,
                        static_cast<uint32_t>(m), static_cast<uint32_t>(n));
}

uint64_t bwg_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes, int swizzle) {
  return make_smem_desc(smem_addr, lbo_bytes, sbo_bytes, static_cast<uint32_t>(swizzle));
}

uint32_t bwg_swizzle128_offset(uint32_t row, uint32_t chunk) { return swizzle128_offset(row, chunk); }

void bwg_raster_tile(int t, int num_m_tiles, int num_n_tiles, int group_m, int* m_tile,
                     int* n_tile) {
  raster_tile(t, num_m_tiles, num_n_tiles, group_m, m_tile, n_tile);
}

int bwg_grouped_schedule(const int* offsets, int G, int M_total, int N, int tile_m, int* prefix,
                         int* lo, int* hi) {
  return grouped_tables(offsets, 0, G, G, M_total, ceil_div(N, kTileN), tile_m, prefix, lo, hi) ? 1
                                                                                                 : 0;
}

void bwg_grouped_tile(int t, int G, const int* prefix, const int* lo, const int* hi, int tile_m,
                      int* g, int* m0, int* n0, int* row_end) {
  grouped_tile(t, G, prefix, lo, hi, tile_m, kTileN, g, m0, n0, row_end);
}

int bwg_tail_split(int T, int C) { return tail_split_count(T, C); }

int bwg_tail_split_f(int T, int C, int max_f, int* f) {
  return tail_split(T, C, max_f, max_f == 4 ? kCostHalf2 : kCostHalf1, kCostQuarter2, f);
}

int bwg_streamk_tiles(int T, int C, int kb, int cut_cost, int* segs) {
  return streamk_tiles(T, C, kb, cut_cost, segs);
}

void bwg_unit_part(int u, int T, int R, int f, int* tile, int* part, int* parts) {
  unit_part(u, T, R, f, tile, part, parts);
}

void bwg_unit_tile(int u, int T, int R, int tile_n, int* tile, int* col_off, int* width) {
  unit_tile(u, T, R, tile_n, tile, col_off, width);
}

long long bwg_streamk_begin(int i, long long W, int C) { return streamk_begin(i, W, C); }

void bwg_streamk_tile_workers(int t, int kb, long long W, int C, int* first, int* count) {
  streamk_tile_workers(t, kb, W, C, first, count);
}

int bwg_grouped_swap_rows(int m0, int row_end, int tile_m) {
  return grouped_swap_rows(m0, row_end, tile_m);
}

#ifndef BWG_SOURCE_HASH
#define BWG_SOURCE_HASH "unknown"
#endif
// The build passes the hash of the library's sources (code only, comments
// and blank space removed), so that a loaded binary can be matched to them.
const char* bwg_version(void) { return "bwgemm 0.2 (sm_103a) source " BWG_SOURCE_HASH; }

}  // extern "C"
