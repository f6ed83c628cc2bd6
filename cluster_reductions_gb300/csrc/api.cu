// api.cu -- the C ABI of librr.so (declared in include/rr.h): argument
// validation, tier dispatch, device-property cache and the device error word.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
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

int occupancy_clusters(const void *func, int threads, size_t smem, int cluster, int device) {
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

bool log_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("RR_LOG");
    return v && *v && std::strcmp(v, "0") != 0;
  }();
  return on;
}

const DevInfo *current_device(int *status) {
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

int rr_plan_reduce(int64_t rows, int64_t cols, int sm_count, int max_cluster, int *tier_out,
                   int *cluster_out) {
  if (rows < 0 || cols < 0 || sm_count < 1 || !tier_out || !cluster_out) return RR_ERR_INVALID;
  int tier = RR_TIER_BLOCK, C = 1;
  if (cols <= 16) {
    tier = RR_TIER_TILED;
  } else if (cols <= 32) {
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
  if (o.tier == RR_TIER_WARP && cols > 32) return RR_ERR_INVALID;
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

static bool rowwise_opts_ok(const rr_rowwise_opts *o) {
  if (!o) return true;
  if (!(o->tier == RR_TIER_AUTO || o->tier == RR_TIER_BLOCK || o->tier == RR_TIER_SPLITK))
    return false;
  return o->cluster_size == 0 || o->cluster_size == 1 || o->cluster_size == 2 ||
         o->cluster_size == 4 || o->cluster_size == 8 || o->cluster_size == 16;
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
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_softmax(x, rows, cols, in_dtype, out, as_stream(stream), *d, &tier,
                      opts ? opts->tier : RR_TIER_AUTO, opts ? opts->cluster_size : 0);
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
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_layernorm_stats(x, rows, cols, in_dtype, eps, mean, rstd, as_stream(stream), *d,
                              &tier, opts ? opts->tier : RR_TIER_AUTO,
                              opts ? opts->cluster_size : 0);
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
  int st = RR_OK;
  const DevInfo *d = current_device(&st);
  if (!d) return st;
  int tier = RR_TIER_BLOCK;
  st = launch_layernorm(x, rows, cols, in_dtype, eps, gamma, beta, out_bf16, mean, rstd,
                        as_stream(stream), *d, &tier, opts ? opts->tier : RR_TIER_AUTO,
                        opts ? opts->cluster_size : 0);
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
  if (P > 1 && !d->cluster_launch) return RR_ERR_UNSUPPORTED;
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
