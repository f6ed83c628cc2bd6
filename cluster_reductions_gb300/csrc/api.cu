// api.cu -- the C ABI of librr.so (declared in include/rr.h): argument
// validation, tier dispatch, device-property cache and the device error word.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <unordered_map>

#include "rr.h"
#include "rr_internal.h"

namespace rr {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
std::atomic<int> g_last_tier{0};

// Split-K cluster-size support, cached per (device, op, dtype).
int g_max_cluster[kMaxDevices][3][2];
bool g_max_cluster_known[kMaxDevices][3][2];

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x0 = (uintptr_t)a, x1 = x0 + na, y0 = (uintptr_t)b, y1 = y0 + nb;
  return na > 0 && nb > 0 && x0 < y1 && y0 < x1;
}

bool mul_overflows(int64_t a, int64_t b, int64_t limit) {
  return a > 0 && b > limit / a;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }
}  // namespace

int cuda_status(cudaError_t e) { return e == cudaSuccess ? RR_OK : RR_ERR_CUDA; }

namespace {
struct OccKey {
  const void *func;
  int threads, cluster, device;
  size_t smem;
  bool operator==(const OccKey &o) const {
    return func == o.func && threads == o.threads && cluster == o.cluster && device == o.device &&
           smem == o.smem;
  }
};
struct OccHash {
  size_t operator()(const OccKey &k) const {
    return std::hash<const void *>()(k.func) ^ ((size_t)k.threads << 20) ^
           ((size_t)k.cluster << 40) ^ ((size_t)k.device << 48) ^ (k.smem * 2654435761u);
  }
};
std::mutex g_occ_mu;
std::unordered_map<OccKey, int, OccHash> g_occ;
}  // namespace

int occupancy_blocks(const void *func, int threads, size_t smem, int device) {
  const OccKey key{func, threads, 0, device, smem};
  {
    std::lock_guard<std::mutex> lock(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, func, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    nb = 0;
  }
  if (nb < 1) nb = 1;
  std::lock_guard<std::mutex> lock(g_occ_mu);
  g_occ[key] = nb;
  return nb;
}

int cluster_cap() {
  static const int cap = [] {
    const char *v = std::getenv("RR_MAX_CLUSTER");
    if (!v || !*v) return 16;
    const int c = std::atoi(v);
    return c < 1 ? 1 : (c > 16 ? 16 : c);
  }();
  return cap;
}

int occupancy_clusters(const void *func, int threads, size_t smem, int cluster, int device) {
  if (cluster > cluster_cap()) return 0;
  const OccKey key{func, threads, cluster, device, smem};
  {
    std::lock_guard<std::mutex> lock(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(g_occ_mu);
  g_occ[key] = n;
  return n;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("RR_PDL");
    return !(v && std::strcmp(v, "0") == 0);
  }();
  return on;
}

bool log_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("RR_LOG");
    return v && *v && std::strcmp(v, "0") != 0;
  }();
  return on;
}

namespace {
std::atomic<int> g_inject_errors{0};
}  // namespace

const DevInfo *current_device(int *status) {
  // failure injection for tests: fail before touching the device
  for (int n = g_inject_errors.load(); n > 0; n = g_inject_errors.load()) {
    if (g_inject_errors.compare_exchange_weak(n, n - 1)) {
      *status = RR_ERR_CUDA;
      return nullptr;
    }
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = RR_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo &d = g_dev[dev];
  if (d.device < 0) {
    DevInfo n;
    n.device = dev;
    if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&n.cluster_launch, cudaDevAttrClusterLaunch, dev) != cudaSuccess) {
      cudaGetLastError();
      *status = RR_ERR_CUDA;
      return nullptr;
    }
    void *w = nullptr;
    if (cudaMalloc(&w, sizeof(int)) != cudaSuccess || cudaMemset(w, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      *status = RR_ERR_CUDA;
      return nullptr;
    }
    n.err_word = (int *)w;
    d = n;
  }
  *status = RR_OK;
  return &d;
}

static int max_cluster_cached(int op, int dtype, const DevInfo &d) {
  const int di = dtype == RR_I32 ? 1 : 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_max_cluster_known[d.device][op][di]) return g_max_cluster[d.device][op][di];
  }
  const int c = d.cluster_launch ? splitk_max_cluster(op, dtype, 16, d) : 1;
  std::lock_guard<std::mutex> lock(g_mu);
  g_max_cluster[d.device][op][di] = c;
  g_max_cluster_known[d.device][op][di] = true;
  return c;
}

}  // namespace rr

using namespace rr;

extern "C" {

const char *rr_status_string(int status) {
  switch (status) {
    case RR_OK: return "ok";
    case RR_ERR_INVALID: return "invalid argument";
    case RR_ERR_UNSUPPORTED: return "unsupported on this device";
    case RR_ERR_CUDA: return "CUDA runtime error";
    case RR_ERR_TIMEOUT: return "device wait timed out";
    case RR_ERR_MISMATCH: return "self-test mismatch";
    default: return "unknown status";
  }
}

int rr_last_tier(void) { return g_last_tier.load(); }

int rr_test_inject_error(int count) {
  if (count < 0) return RR_ERR_INVALID;
  g_inject_errors.store(count);
  return RR_OK;
}

int rr_plan_reduce(int64_t rows, int64_t cols, int sm_count, int max_cluster, int *tier_out,
                   int *cluster_out) {
  if (rows < 0 || cols < 0 || sm_count < 1 || !tier_out || !cluster_out) return RR_ERR_INVALID;
  int tier = RR_TIER_BLOCK, C = 1;
  if (cols <= 32) {
    // rows of up to 32 elements: a thread per row (tiled), except 16 and
    // 29-32, where a warp's lanes split the row (measured: 16 columns 6858
    // against 6425 GB/s, 32 6893 against 5697; 20-28 the other way round,
    // 6161 against 3199 for 24)
    tier = (cols == 16 || cols >= 29) ? RR_TIER_WARP : RR_TIER_TILED;
  } else if (cols < 4096 && rows >= sm_count) {
    // warp segments per row: rows too short for a CTA each, enough of them
    // to fill the GPU
    tier = RR_TIER_WARP;
  } else if (rows >= 1 && rows < sm_count && cols >= 4096 && max_cluster >= 2) {
    // the smallest power of two that puts at least one CTA on every SM,
    // capped by 16 and by what the device can co-schedule
    const int cap = max_cluster < 16 ? max_cluster : 16;
    int c = 2;
    while (c < cap && (int64_t)c * rows < sm_count) c *= 2;
    tier = RR_TIER_SPLITK;
    C = c;
  }
  *tier_out = tier;
  *cluster_out = C;
  return RR_OK;
}

int rr_plan_rowwise(int64_t rows, int64_t cols, int in_dtype, int row_op, int aligned,
                    int sm_count, int max_cluster, int with_workspace, int *tier_out,
                    int *width_out, int *staged_out) {
  if (rows < 0 || cols < 0 || sm_count < 1 || max_cluster < 1 || !tier_out || !width_out)
    return RR_ERR_INVALID;
  if (in_dtype != RR_BF16 && in_dtype != RR_F32) return RR_ERR_INVALID;
  if (row_op < RR_ROW_SOFTMAX || row_op > RR_ROW_LAYERNORM) return RR_ERR_INVALID;
  const int epv = in_dtype == RR_BF16 ? 8 : 4;
  const bool vec = aligned && cols % epv == 0;
  const bool half = aligned && cols % (epv / 2) == 0;  // 8-byte vectors
  const RowPlan p = plan_rowwise(rows, cols, in_dtype, vec, row_op, RR_TIER_AUTO, 0, sm_count,
                                 max_cluster < 16 ? max_cluster : 16, true, half,
                                 with_workspace != 0 && vec);
  *tier_out = p.tier;
  *width_out = p.width;
  if (staged_out)
    *staged_out = p.twopass ? 5 : (p.chunk ? 4 : (p.grid ? 3 : (p.ring ? 2 : (p.staged ? 1 : 0))));
  return RR_OK;
}

int rr_rowwise_workspace_size(int64_t rows, int64_t cols, int in_dtype, int row_op,
                              size_t *bytes_out) {
  if (rows < 0 || cols < 0 || !bytes_out) return RR_ERR_INVALID;
  if (in_dtype != RR_BF16 && in_dtype != RR_F32) return RR_ERR_INVALID;
  if (row_op < RR_ROW_SOFTMAX || row_op > RR_ROW_LAYERNORM) return RR_ERR_INVALID;
  *bytes_out = 0;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  const int cap = cluster_cap() < 16 ? cluster_cap() : 16;
  int tier = 0, width = 0, staged = 0;
  st = rr_plan_rowwise(rows, cols, in_dtype, row_op, 1, d->sm_count, d->cluster_launch ? cap : 1,
                       1, &tier, &width, &staged);
  if (st != RR_OK) return st;
  if (staged == 3) *bytes_out = rowgrid_ws_bytes(rows, width);
  if (staged == 5) *bytes_out = rowtwopass_ws_bytes(rows);
  return RR_OK;
}

int rr_reduce_ex(const void *x, int64_t rows, int64_t cols, int op, int dtype, void *out,
                 void *stream, const rr_reduce_opts *opts) {
  if (rows < 0 || cols < 0) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN) return RR_ERR_INVALID;
  if (dtype != RR_F32 && dtype != RR_I32) return RR_ERR_INVALID;
  rr_reduce_opts o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.tier < RR_TIER_AUTO || o.tier > RR_TIER_SPLITK) return RR_ERR_INVALID;
  if (!(o.cluster_size == 0 || o.cluster_size == 1 || o.cluster_size == 2 ||
        o.cluster_size == 4 || o.cluster_size == 8 || o.cluster_size == 16))
    return RR_ERR_INVALID;
  if (!(o.emit_tile_width == 0 || o.emit_tile_width == 1 || o.emit_tile_width == 2 ||
        o.emit_tile_width == 4))
    return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (!out || (cols > 0 && !x)) return RR_ERR_INVALID;
  if (mul_overflows(rows, cols, INT64_MAX / 4)) return RR_ERR_INVALID;
  if (overlaps(x, (size_t)(rows * cols * 4), out, (size_t)rows * 4)) return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = o.tier, C = o.cluster_size;
  if (tier == RR_TIER_AUTO) {
    const int maxc = max_cluster_cached(op, dtype, *d);
    int auto_c = 1;
    rr_plan_reduce(rows, cols, d->sm_count, maxc, &tier, &auto_c);
    if (C == 0) C = auto_c;
  }
  if (tier == RR_TIER_SPLITK) {
    if (C == 0) {
      const int maxc = max_cluster_cached(op, dtype, *d);
      const int cap = maxc < 16 ? maxc : 16;
      C = 1;
      while (C < cap && (int64_t)C * rows < d->sm_count) C *= 2;
    }
    if (C > 1 && (!d->cluster_launch || max_cluster_cached(op, dtype, *d) < C))
      return RR_ERR_UNSUPPORTED;
    if (rows > INT_MAX / C) return RR_ERR_INVALID;
    if (o.rank_out && overlaps(o.rank_out, (size_t)(rows * C * 4), x, (size_t)(rows * cols * 4)))
      return RR_ERR_INVALID;
  } else {
    C = 1;
  }
  st = launch_reduce(x, rows, cols, op, dtype, out, as_stream(stream), tier, C,
                     o.emit_tile_width, tier == RR_TIER_SPLITK ? o.rank_out : nullptr, *d);
  if (st == RR_OK) g_last_tier.store((C << 8) | tier);
  return st;
}

int rr_reduce_splitk_multi(const void *x, int64_t rows, int64_t cols, int op, int dtype, void *out,
                           int cluster_size, int clusters_per_row, void *workspace,
                           size_t workspace_bytes, void *stream) {
  if (rows < 0 || cols < 0) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN) return RR_ERR_INVALID;
  if (dtype != RR_F32 && dtype != RR_I32) return RR_ERR_INVALID;
  if (!(cluster_size == 0 || cluster_size == 1 || cluster_size == 2 || cluster_size == 4 ||
        cluster_size == 8 || cluster_size == 16))
    return RR_ERR_INVALID;
  if (clusters_per_row < 0 || clusters_per_row > 1024) return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (!out || !workspace || (cols > 0 && !x)) return RR_ERR_INVALID;
  if (mul_overflows(rows, cols, INT64_MAX / 4)) return RR_ERR_INVALID;
  if (overlaps(x, (size_t)(rows * cols * 4), out, (size_t)rows * 4)) return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  const int maxc = max_cluster_cached(op, dtype, *d);
  int C = cluster_size == 0 ? (maxc < 16 ? maxc : 16) : cluster_size;
  if (C < 1) C = 1;
  if (C > 1 && (!d->cluster_launch || maxc < C)) return RR_ERR_UNSUPPORTED;
  int G = clusters_per_row;
  if (G == 0) {  // enough clusters that every SM holds a CTA
    const int64_t need = (d->sm_count + rows * C - 1) / (rows * C);
    G = (int)(need < 1 ? 1 : (need > 1024 ? 1024 : need));
  }
  if (rows * (int64_t)G * C > INT_MAX) return RR_ERR_INVALID;
  if (workspace_bytes < (size_t)rows * G * 4) return RR_ERR_INVALID;
  if (overlaps(workspace, (size_t)rows * G * 4, x, (size_t)(rows * cols * 4)) ||
      overlaps(workspace, (size_t)rows * G * 4, out, (size_t)rows * 4))
    return RR_ERR_INVALID;
  st = launch_reduce_splitk_multi(x, rows, cols, op, dtype, out, C, G, workspace,
                                  as_stream(stream));
  if (st == RR_OK) g_last_tier.store((C << 8) | RR_TIER_SPLITK);
  return st;
}

int rr_reduce(const void *x, int64_t rows, int64_t cols, int op, int dtype, void *out,
              void *stream) {
  return rr_reduce_ex(x, rows, cols, op, dtype, out, stream, nullptr);
}

// ---------------------------------------------------------------------------
// Reduction over a non-last axis.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {
// Tiles of the warp / block / split-K tiers: (o, L*V adjacent rows).
int64_t axis_units(int64_t outer, int64_t inner, int V, int lg_L) {
  const int64_t TW = ((int64_t)1 << lg_L) * V;
  return outer * ((inner + TW - 1) / TW);
}

// The automatic plan for inner > 1.  Targets (S = SM count):
//  - tiled when there are at least 2048 * S independent row groups: every
//    thread of a full GPU owns rows and no combine is needed;
//  - warp when the full-width tiles number at least 32 * S;
//  - block when they number at least 2 * S, after narrowing the tile (down
//    to 64-byte row segments) to make more of them;
//  - split-K otherwise: the smallest power-of-two cluster giving 2 * S CTAs
//    (at most 16 and what the device co-schedules); if even that falls
//    short and a workspace may be used, clusters of at most 8 CTAs (16-CTA
//    clusters pack less densely onto the SMs) and G of them per tile,
//    enough for 3 * S CTAs, each folding at least 256 axis positions,
//    G <= 1024.
AxisPlan plan_axis(int64_t outer, int64_t axis, int64_t inner, int S, int max_cluster,
                   int x_align, bool with_ws) {
  AxisPlan p;
  // narrow inner widths that are not a multiple of 4: the contiguous slabs
  // x[o, :, :] read with 16-byte loads, a warp per slab when there are at
  // least 16 per SM, a CTA per slab from 2 per SM
  if ((inner == 2 || inner == 3 || inner == 5 || inner == 6 || inner == 7) &&
      x_align % 16 == 0 && (axis * inner) % 4 == 0 && axis >= 4 &&
      outer >= (int64_t)S * 2) {
    p.tier = outer >= (int64_t)S * 16 ? RR_TIER_WARP : RR_TIER_BLOCK;
    p.V = 1;
    p.slab = true;
    return p;
  }
  p.V = (x_align % 16 == 0 && inner % 4 == 0) ? 4 : 1;
  const int E = p.V == 4 ? 4 : ((x_align % 8 == 0 && inner % 2 == 0) ? 2 : 1);
  if (outer * (inner / E) >= (int64_t)S * 2048) {
    p.tier = RR_TIER_TILED;
    p.E = E;
    return p;
  }
  int lg = 0;
  while (lg < 5 && ((int64_t)p.V << lg) < inner) ++lg;
  p.lg_L = lg;
  int64_t units = axis_units(outer, inner, p.V, lg);
  if (units >= (int64_t)S * 32) {
    p.tier = RR_TIER_WARP;
    return p;
  }
  const int lg_min = p.V == 4 ? 2 : 4;  // 64-byte segments
  while (p.lg_L > lg_min && units < (int64_t)S * 2) {
    --p.lg_L;
    units = axis_units(outer, inner, p.V, p.lg_L);
  }
  p.tier = RR_TIER_BLOCK;
  if (units >= (int64_t)S * 2) return p;
  if (max_cluster >= 2) {
    const int cap = max_cluster < 16 ? max_cluster : 16;
    p.tier = RR_TIER_SPLITK;
    p.C = 2;
    while (p.C < cap && units * p.C < (int64_t)S * 2) p.C *= 2;
    if (units * p.C >= (int64_t)S * 2) return p;
  }
  if (!with_ws) return p;
  if (p.C > 8) p.C = 8;
  int64_t G = ((int64_t)S * 3 + units * p.C - 1) / (units * p.C);
  const int64_t gmax = axis / ((int64_t)p.C * 256);
  if (G > gmax) G = gmax;
  if (G > 1024) G = 1024;
  p.G = G < 1 ? 1 : (int)G;
  return p;
}

void plan_to_c(const AxisPlan &p, int64_t outer, int64_t inner, rr_axis_plan *c) {
  c->tier = p.tier;
  c->cluster_size = p.tier == RR_TIER_SPLITK ? p.C : 1;
  c->emit_tile_width = p.tier == RR_TIER_TILED ? p.E : 0;
  c->tile_rows = p.tier == RR_TIER_TILED ? 0 : (p.slab ? (int)inner : (p.V << p.lg_L));
  c->splits = p.G;
  c->workspace_bytes = p.G > 1 ? (size_t)p.G * (size_t)(outer * inner) * 4 : 0;
}

std::mutex g_axis_mu;
int g_axis_maxc[rr::kMaxDevices];
bool g_axis_maxc_known[rr::kMaxDevices];

int axis_max_cluster_cached(const rr::DevInfo &d) {
  std::lock_guard<std::mutex> lock(g_axis_mu);
  if (!g_axis_maxc_known[d.device]) {
    g_axis_maxc[d.device] = rr::axis_max_cluster(16, d);
    g_axis_maxc_known[d.device] = true;
  }
  return g_axis_maxc[d.device];
}

bool axis_sizes_ok(int64_t outer, int64_t axis, int64_t inner) {
  return outer >= 0 && axis >= 0 && inner >= 0 && !mul_overflows(outer, axis, INT64_MAX / 4) &&
         !mul_overflows(outer * axis, inner, INT64_MAX / 4) &&
         !mul_overflows(outer, inner, INT64_MAX / 4096);
}
}  // namespace

extern "C" {

int rr_plan_reduce_axis(int64_t outer, int64_t axis, int64_t inner, int sm_count,
                        int max_cluster, int x_align, int with_workspace, rr_axis_plan *plan) {
  if (!axis_sizes_ok(outer, axis, inner) || sm_count < 1 || !plan ||
      !(x_align == 4 || x_align == 8 || x_align == 16))
    return RR_ERR_INVALID;
  if (inner == 1) {
    std::memset(plan, 0, sizeof(*plan));
    plan->splits = 1;
    return rr_plan_reduce(outer, axis, sm_count, max_cluster, &plan->tier, &plan->cluster_size);
  }
  plan_to_c(plan_axis(outer, axis, inner, sm_count, max_cluster, x_align, with_workspace != 0),
            outer, inner, plan);
  return RR_OK;
}

int rr_reduce_axis_workspace_size(int64_t outer, int64_t axis, int64_t inner, int x_align,
                                  size_t *bytes_out) {
  if (!bytes_out || !axis_sizes_ok(outer, axis, inner) ||
      !(x_align == 4 || x_align == 8 || x_align == 16))
    return RR_ERR_INVALID;
  *bytes_out = 0;
  if (inner <= 1 || outer == 0) return RR_OK;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  rr_axis_plan c;
  plan_to_c(plan_axis(outer, axis, inner, d->sm_count, axis_max_cluster_cached(*d), x_align, true),
            outer, inner, &c);
  *bytes_out = c.workspace_bytes;
  return RR_OK;
}

int rr_reduce_axis_ex(const void *x, int64_t outer, int64_t axis, int64_t inner, int op,
                      int dtype, void *out, void *stream, const rr_axis_opts *opts) {
  if (!axis_sizes_ok(outer, axis, inner)) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN) return RR_ERR_INVALID;
  if (dtype != RR_F32 && dtype != RR_I32) return RR_ERR_INVALID;
  rr_axis_opts o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.tier < RR_TIER_AUTO || o.tier > RR_TIER_SPLITK) return RR_ERR_INVALID;
  if (!(o.cluster_size == 0 || o.cluster_size == 1 || o.cluster_size == 2 ||
        o.cluster_size == 4 || o.cluster_size == 8 || o.cluster_size == 16))
    return RR_ERR_INVALID;
  if (!(o.emit_tile_width == 0 || o.emit_tile_width == 1 || o.emit_tile_width == 2 ||
        o.emit_tile_width == 4))
    return RR_ERR_INVALID;
  if (o.tile_rows < 0 || o.tile_rows > 128 || (o.tile_rows & (o.tile_rows - 1)) != 0)
    return RR_ERR_INVALID;
  if (o.splits < 0 || o.splits > 65536) return RR_ERR_INVALID;
  if (inner == 1) {
    if (o.tile_rows != 0 || o.splits > 1) return RR_ERR_INVALID;
    rr_reduce_opts ro;
    std::memset(&ro, 0, sizeof(ro));
    ro.tier = o.tier;
    ro.cluster_size = o.cluster_size;
    ro.emit_tile_width = o.emit_tile_width;
    return rr_reduce_ex(x, outer, axis, op, dtype, out, stream, &ro);
  }
  if (outer == 0 || inner == 0) return RR_OK;
  const int64_t nx = outer * axis * inner, nout = outer * inner;
  if (!out || (nx > 0 && !x)) return RR_ERR_INVALID;
  if (overlaps(x, (size_t)nx * 4, out, (size_t)nout * 4)) return RR_ERR_INVALID;
  if (((uintptr_t)x & 3u) != 0) return RR_ERR_INVALID;
  const bool have_ws = o.workspace != nullptr && o.workspace_bytes > 0;
  if (have_ws && (overlaps(o.workspace, o.workspace_bytes, x, (size_t)nx * 4) ||
                  overlaps(o.workspace, o.workspace_bytes, out, (size_t)nout * 4)))
    return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  const int x_align = ((uintptr_t)x & 15u) == 0 ? 16 : (((uintptr_t)x & 7u) == 0 ? 8 : 4);
  const int maxc = d->cluster_launch ? axis_max_cluster_cached(*d) : 1;
  AxisPlan p = plan_axis(outer, axis, inner, d->sm_count, maxc, x_align, have_ws);
  if (o.tier != RR_TIER_AUTO && o.tier != p.tier) {
    // a forced tier: its own defaults, from the same rules
    AxisPlan f;
    f.tier = o.tier;
    f.V = p.V;
    int lg = 0;
    while (lg < 5 && ((int64_t)f.V << lg) < inner) ++lg;
    f.lg_L = lg;
    if (o.tier == RR_TIER_TILED) {
      f.E = f.V == 4 ? 4 : ((x_align >= 8 && inner % 2 == 0) ? 2 : 1);
    } else if (o.tier == RR_TIER_SPLITK) {
      const int64_t units = axis_units(outer, inner, f.V, f.lg_L);
      const int cap = maxc < 16 ? maxc : 16;
      f.C = cap < 2 ? 1 : 2;
      while (f.C < cap && units * f.C < (int64_t)d->sm_count * 2) f.C *= 2;
    }
    p = f;
  }
  if (p.tier == RR_TIER_TILED) {
    if (o.emit_tile_width) p.E = o.emit_tile_width;
    if ((p.E == 4 && !(x_align == 16 && inner % 4 == 0)) ||
        (p.E == 2 && !(x_align >= 8 && inner % 2 == 0)))
      return RR_ERR_INVALID;
    p.C = 1;
    p.G = 1;
  } else {
    if (o.tile_rows) {
      if (o.tile_rows % p.V != 0 || o.tile_rows / p.V > 32) return RR_ERR_INVALID;
      int lg = 0;
      while ((p.V << lg) < o.tile_rows) ++lg;
      p.lg_L = lg;
    }
    if (p.tier == RR_TIER_SPLITK) {
      if (o.cluster_size) p.C = o.cluster_size;
      if (p.C > 1 && (!d->cluster_launch || maxc < p.C)) return RR_ERR_UNSUPPORTED;
    } else {
      p.C = 1;
    }
    if (p.tier == RR_TIER_WARP) p.G = 1;
    if (o.splits) {
      if (p.tier == RR_TIER_WARP && o.splits > 1) return RR_ERR_INVALID;
      p.G = o.splits;
    }
    if (p.G > 1) {
      if (!have_ws || o.workspace_bytes / 4 / (size_t)p.G < (size_t)nout) return RR_ERR_INVALID;
      if (((uintptr_t)o.workspace & 3u) != 0) return RR_ERR_INVALID;
      if (axis_units(outer, inner, p.V, p.lg_L) * p.G > ((int64_t)1 << 40)) return RR_ERR_INVALID;
    }
  }
  st = launch_reduce_axis(x, outer, axis, inner, op, dtype, out, p, o.workspace,
                          as_stream(stream), *d);
  if (st == RR_OK) g_last_tier.store((p.C << 8) | p.tier);
  return st;
}

int rr_reduce_axis(const void *x, int64_t outer, int64_t axis, int64_t inner, int op, int dtype,
                   void *out, void *stream) {
  return rr_reduce_axis_ex(x, outer, axis, inner, op, dtype, out, stream, nullptr);
}

static bool rowwise_opts_ok(const rr_rowwise_opts *o) {
  if (!o) return true;
  if (!(o->tier == RR_TIER_AUTO || o->tier == RR_TIER_WARP || o->tier == RR_TIER_BLOCK ||
        o->tier == RR_TIER_SPLITK))
    return false;
  const int l = o->lanes_per_row;
  if (!(l == 0 || l == 1 || l == 2 || l == 4 || l == 8 || l == 16 || l == 32)) return false;
  if (!(o->cluster_size == 0 || o->cluster_size == 1 || o->cluster_size == 2 ||
        o->cluster_size == 4 || o->cluster_size == 8 || o->cluster_size == 16))
    return false;
  // the grid form: forced only as split-K without a cluster, with a workspace
  if (o->splits < 0 || o->splits > kRowGridMaxSplits) return false;
  if (o->splits > 0 && (o->tier != RR_TIER_SPLITK || o->cluster_size > 1 || !o->workspace))
    return false;
  if (o->workspace && (o->workspace_bytes == 0 || (uintptr_t)o->workspace % 16 != 0)) return false;
  return true;
}

// The caller's workspace of a row op, and whether it overlaps any operand.
static RowWs rowwise_ws(const rr_rowwise_opts *o) {
  RowWs w;
  if (o) {
    w.ws = o->workspace;
    w.bytes = o->workspace ? o->workspace_bytes : 0;
    w.splits = o->splits;
  }
  return w;
}
struct Span {
  const void *p;
  size_t n;
};
static bool ws_overlaps(const RowWs &w, std::initializer_list<Span> spans) {
  if (!w.ws) return false;
  for (const Span &sp : spans)
    if (sp.p && overlaps(w.ws, w.bytes, sp.p, sp.n)) return true;
  return false;
}

// The width a forced row-op tier takes: lanes per row for the warp tier, the
// cluster size otherwise.
static int rowwise_width(const rr_rowwise_opts *o) {
  if (!o) return 0;
  return o->tier == RR_TIER_WARP ? o->lanes_per_row : o->cluster_size;
}

int rr_softmax(const void *x, int64_t rows, int64_t cols, int in_dtype, float *out,
               void *stream) {
  return rr_softmax_ex(x, rows, cols, in_dtype, out, stream, nullptr);
}

int rr_softmax_ex(const void *x, int64_t rows, int64_t cols, int in_dtype, float *out,
                  void *stream, const rr_rowwise_opts *opts) {
  if (!rowwise_opts_ok(opts)) return RR_ERR_INVALID;
  if (rows < 0 || cols < 0) return RR_ERR_INVALID;
  if (in_dtype != RR_BF16 && in_dtype != RR_F32) return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (cols == 0 || !x || !out) return RR_ERR_INVALID;
  if (mul_overflows(rows, cols, INT64_MAX / 4)) return RR_ERR_INVALID;
  const size_t es = in_dtype == RR_BF16 ? 2 : 4;
  if (overlaps(x, (size_t)(rows * cols) * es, out, (size_t)(rows * cols) * 4)) return RR_ERR_INVALID;
  if ((uintptr_t)x % es != 0 || (uintptr_t)out % 4 != 0) return RR_ERR_INVALID;
  const RowWs w = rowwise_ws(opts);
  if (ws_overlaps(w, {{x, (size_t)(rows * cols) * es}, {out, (size_t)(rows * cols) * 4}}))
    return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_softmax(x, rows, cols, in_dtype, out, as_stream(stream), *d, &tier,
                      opts ? opts->tier : RR_TIER_AUTO, rowwise_width(opts), w);
  if (st == RR_OK) g_last_tier.store(tier);
  return st;
}

int rr_layernorm_stats(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                       float *mean, float *rstd, void *stream) {
  return rr_layernorm_stats_ex(x, rows, cols, in_dtype, eps, mean, rstd, stream, nullptr);
}

int rr_layernorm_stats_ex(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                          float *mean, float *rstd, void *stream, const rr_rowwise_opts *opts) {
  if (!rowwise_opts_ok(opts)) return RR_ERR_INVALID;
  if (rows < 0 || cols < 0) return RR_ERR_INVALID;
  if (in_dtype != RR_BF16 && in_dtype != RR_F32) return RR_ERR_INVALID;
  if (!(eps >= 0.0f) || std::isinf(eps)) return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (cols == 0 || !x || !mean || !rstd) return RR_ERR_INVALID;
  if (mul_overflows(rows, cols, INT64_MAX / 4)) return RR_ERR_INVALID;
  const size_t es = in_dtype == RR_BF16 ? 2 : 4;
  const size_t nx = (size_t)(rows * cols) * es, no = (size_t)rows * 4;
  if (overlaps(x, nx, mean, no) || overlaps(x, nx, rstd, no) || overlaps(mean, no, rstd, no))
    return RR_ERR_INVALID;
  if ((uintptr_t)x % es != 0) return RR_ERR_INVALID;
  const RowWs w = rowwise_ws(opts);
  if (ws_overlaps(w, {{x, nx}, {mean, no}, {rstd, no}})) return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_layernorm_stats(x, rows, cols, in_dtype, eps, mean, rstd, as_stream(stream), *d,
                              &tier, opts ? opts->tier : RR_TIER_AUTO,
                              rowwise_width(opts), w);
  if (st == RR_OK) g_last_tier.store(tier);
  return st;
}

int rr_layernorm(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                 const float *gamma, const float *beta, uint16_t *out_bf16, float *mean,
                 float *rstd, void *stream) {
  return rr_layernorm_ex(x, rows, cols, in_dtype, eps, gamma, beta, out_bf16, mean, rstd, stream,
                         nullptr);
}

int rr_layernorm_ex(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                    const float *gamma, const float *beta, uint16_t *out_bf16, float *mean,
                    float *rstd, void *stream, const rr_rowwise_opts *opts) {
  if (!rowwise_opts_ok(opts)) return RR_ERR_INVALID;
  if (rows < 0 || cols < 0) return RR_ERR_INVALID;
  if (in_dtype != RR_BF16 && in_dtype != RR_F32) return RR_ERR_INVALID;
  if (!(eps >= 0.0f) || std::isinf(eps)) return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (cols == 0 || !x || !gamma || !beta || !out_bf16) return RR_ERR_INVALID;
  if (mul_overflows(rows, cols, INT64_MAX / 4)) return RR_ERR_INVALID;
  const size_t es = in_dtype == RR_BF16 ? 2 : 4;
  const size_t nx = (size_t)(rows * cols) * es, ny = (size_t)(rows * cols) * 2,
               no = (size_t)rows * 4, ng = (size_t)cols * 4;
  if (overlaps(x, nx, out_bf16, ny) || overlaps(gamma, ng, out_bf16, ny) ||
      overlaps(beta, ng, out_bf16, ny))
    return RR_ERR_INVALID;
  if ((mean && (overlaps(mean, no, out_bf16, ny) || overlaps(mean, no, x, nx))) ||
      (rstd && (overlaps(rstd, no, out_bf16, ny) || overlaps(rstd, no, x, nx))) ||
      (mean && rstd && overlaps(mean, no, rstd, no)))
    return RR_ERR_INVALID;
  if ((uintptr_t)x % es != 0 || (uintptr_t)gamma % 4 || (uintptr_t)beta % 4 ||
      (uintptr_t)out_bf16 % 2)
    return RR_ERR_INVALID;
  const RowWs w = rowwise_ws(opts);
  if (ws_overlaps(w, {{x, nx}, {out_bf16, ny}, {gamma, ng}, {beta, ng}, {mean, no}, {rstd, no}}))
    return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_layernorm(x, rows, cols, in_dtype, eps, gamma, beta, out_bf16, mean, rstd,
                        as_stream(stream), *d, &tier, opts ? opts->tier : RR_TIER_AUTO,
                        rowwise_width(opts), w);
  if (st == RR_OK) g_last_tier.store(tier);
  return st;
}

int rr_cluster_allreduce(const void *vals, int clusters, int cluster_size, int width, int op,
                         int dtype, int iters, int two_slot, int64_t skew_cycles, void *res,
                         int64_t *mismatches, void *stream) {
  if (clusters < 1 || cluster_size < 1 || cluster_size > 16) return RR_ERR_INVALID;
  if (!(width == 1 || width == 2 || width == 4 || width == 8)) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN) return RR_ERR_INVALID;
  if (dtype != RR_F32 && dtype != RR_I32) return RR_ERR_INVALID;
  if (iters < 0 || skew_cycles < 0 || skew_cycles > (1 << 20)) return RR_ERR_INVALID;
  if ((int64_t)clusters * cluster_size > INT_MAX) return RR_ERR_INVALID;
  if (iters == 0) return RR_OK;
  if (!vals || !res) return RR_ERR_INVALID;
  if (mul_overflows((int64_t)iters, (int64_t)clusters * cluster_size * width, INT64_MAX / 4))
    return RR_ERR_INVALID;
  const size_t n = (size_t)iters * clusters * cluster_size * width * 4;
  if (overlaps(vals, n, res, n)) return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  if (cluster_size > 1 && !d->cluster_launch) return RR_ERR_UNSUPPORTED;
  return launch_cluster_allreduce(vals, clusters, cluster_size, width, op, dtype, iters,
                                  two_slot ? 1 : 0, skew_cycles, res, mismatches,
                                  as_stream(stream), *d);
}

int rr_cluster_allreduce_selftest(int cluster_size, int width, int op, int dtype, int iters,
                                  int two_slot, uint64_t seed, void *stream,
                                  int64_t *mismatches_out) {
  return rr_cluster_allreduce_selftest_ex(cluster_size, width, op, dtype, iters, two_slot, seed,
                                          stream, mismatches_out, nullptr, nullptr);
}

int rr_cluster_allreduce_selftest_ex(int cluster_size, int width, int op, int dtype, int iters,
                                     int two_slot, uint64_t seed, void *stream,
                                     int64_t *mismatches_out, void *vals_host, void *res_host) {
  if (!mismatches_out) return RR_ERR_INVALID;
  if (iters < 1 || iters > (1 << 20)) return RR_ERR_INVALID;
  if (cluster_size < 1 || cluster_size > 16) return RR_ERR_INVALID;
  if (!(width == 1 || width == 2 || width == 4 || width == 8)) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN || (dtype != RR_F32 && dtype != RR_I32))
    return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  const int clusters = 2;
  const int64_t n = (int64_t)iters * clusters * cluster_size * width;
  void *vals = nullptr, *res = nullptr, *mism = nullptr;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMalloc(&vals, (size_t)n * 4);
  if (e == cudaSuccess) e = cudaMalloc(&res, (size_t)n * 4);
  if (e == cudaSuccess) e = cudaMalloc(&mism, sizeof(int64_t));
  if (e == cudaSuccess) e = cudaMemsetAsync(mism, 0, sizeof(int64_t), s);
  if (e != cudaSuccess) {
    st = RR_ERR_CUDA;
  } else {
    st = launch_fill_selftest_values(vals, n, dtype, seed, s);
    if (st == RR_OK)
      st = launch_cluster_allreduce(vals, clusters, cluster_size, width, op, dtype, iters,
                                    two_slot ? 1 : 0, 2000, res, (int64_t *)mism, s, *d);
    int64_t h = -1;
    if (st == RR_OK) {
      if (cudaMemcpyAsync(&h, mism, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          (vals_host && cudaMemcpyAsync(vals_host, vals, (size_t)n * 4, cudaMemcpyDeviceToHost,
                                        s) != cudaSuccess) ||
          (res_host && cudaMemcpyAsync(res_host, res, (size_t)n * 4, cudaMemcpyDeviceToHost,
                                       s) != cudaSuccess) ||
          cudaStreamSynchronize(s) != cudaSuccess)
        st = RR_ERR_CUDA;
    }
    if (st == RR_OK) {
      *mismatches_out = h;
      if (h != 0) st = RR_ERR_MISMATCH;
    }
  }
  cudaStreamSynchronize(s);
  if (vals) cudaFree(vals);
  if (res) cudaFree(res);
  if (mism) cudaFree(mism);
  cudaGetLastError();
  return st;
}

int rr_splitk_combine(const float *O, const float *m, const float *l, int P, int64_t rows, int D,
                      float scale_log2e, uint16_t *out_bf16, void *stream) {
  return rr_splitk_combine_ex(O, m, l, P, rows, D, scale_log2e, out_bf16, stream,
                              RR_COMBINE_AUTO);
}

int rr_splitk_combine_ex(const float *O, const float *m, const float *l, int P, int64_t rows,
                         int D, float scale_log2e, uint16_t *out_bf16, void *stream, int mode) {
  if (P < 1 || P > 16 || rows < 0 || D < 1 || D > 1024) return RR_ERR_INVALID;
  if (mode < RR_COMBINE_AUTO || mode > RR_COMBINE_DIRECT) return RR_ERR_INVALID;
  if (!std::isfinite(scale_log2e)) return RR_ERR_INVALID;
  if (rows == 0) return RR_OK;
  if (!O || !m || !l || !out_bf16) return RR_ERR_INVALID;
  if (mul_overflows((int64_t)P * rows, D, INT64_MAX / 4)) return RR_ERR_INVALID;
  const size_t nO = (size_t)P * rows * D * 4, nml = (size_t)P * rows * 4,
               nout = (size_t)rows * D * 2;
  if (overlaps(O, nO, out_bf16, nout) || overlaps(m, nml, out_bf16, nout) ||
      overlaps(l, nml, out_bf16, nout))
    return RR_ERR_INVALID;
  if ((uintptr_t)O % 4 || (uintptr_t)m % 4 || (uintptr_t)l % 4 || (uintptr_t)out_bf16 % 2)
    return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  return launch_combine(O, m, l, P, rows, D, scale_log2e, out_bf16, as_stream(stream), *d, mode);
}

int rr_device_status(void *stream) {
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return RR_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, d->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RR_ERR_CUDA;
  if (h != 0) {
    if (cudaMemset(d->err_word, 0, sizeof(int)) != cudaSuccess) return RR_ERR_CUDA;
    return RR_ERR_TIMEOUT;
  }
  return RR_OK;
}

int rr_test_wait_timeout(int64_t budget_iters, void *stream) {
  if (budget_iters < 0 || budget_iters > (int64_t(1) << 30)) return RR_ERR_INVALID;
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  return launch_wait_timeout_probe(budget_iters, as_stream(stream), *d);
}

}  // extern "C"
