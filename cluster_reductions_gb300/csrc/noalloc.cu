// noalloc.cu -- the cluster all-reduce self-test without any device
// allocation.  rr_cluster_allreduce_selftest allocates its scratch (the
// seeded per-rank values, the per-rank results and a mismatch counter) with
// cudaMalloc and frees it again.  Some callers cannot do that: a serving
// process whose memory pool has already reserved the whole device, or one
// that must not take the implicit device synchronisation a cudaMalloc /
// cudaFree may cause in the middle of its work.  This variant runs the same
// self-test out of a fixed, file-scope device array instead.
#include <mutex>

#include "rr.h"
#include "rr_internal.h"

namespace rr {
namespace {

// Capacity of the static scratch, in 32-bit values per buffer.  The array
// holds the values buffer, the results buffer and an 8-byte counter, about
// 2 MiB in all; every GPU that loads librr.so keeps it until the process
// exits.
constexpr int64_t kNoAllocMaxValues = int64_t(1) << 18;
constexpr size_t kNoAllocBytes = 2 * (size_t)kNoAllocMaxValues * 4 + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
// Held for a whole self-test: every call uses the same scratch, so calls
// from several host threads run one after another (each is blocking anyway).
std::mutex g_noalloc_run_mu;
void *g_noalloc_ptr[kMaxDev];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device.  The symbol
// name is only a host-side stand-in; the address is looked up once per
// device, with that device current.
int scratch_address(int dev, unsigned char **out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return RR_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<unsigned char *>(g_noalloc_ptr[dev]);
  return RR_OK;
}

}  // namespace
}  // namespace rr

using namespace rr;

extern "C" int rr_cluster_allreduce_selftest_noalloc(int cluster_size, int width, int op,
                                                     int dtype, int iters, int two_slot,
                                                     uint64_t seed, void *stream,
                                                     int64_t *mismatches_out) {
  return rr_cluster_allreduce_selftest_noalloc_ex(cluster_size, width, op, dtype, iters, two_slot,
                                                  seed, stream, mismatches_out, nullptr, nullptr);
}

extern "C" int rr_cluster_allreduce_selftest_noalloc_ex(int cluster_size, int width, int op,
                                                        int dtype, int iters, int two_slot,
                                                        uint64_t seed, void *stream,
                                                        int64_t *mismatches_out, void *vals_host,
                                                        void *res_host) {
  if (!mismatches_out) return RR_ERR_INVALID;
  if (iters < 1 || cluster_size < 1 || cluster_size > 16) return RR_ERR_INVALID;
  if (!(width == 1 || width == 2 || width == 4 || width == 8)) return RR_ERR_INVALID;
  if (op < RR_OP_SUM || op > RR_OP_MIN || (dtype != RR_F32 && dtype != RR_I32))
    return RR_ERR_INVALID;
  const int clusters = 2;
  const int64_t n = (int64_t)iters * clusters * cluster_size * width;
  if (n > kNoAllocMaxValues) return RR_ERR_INVALID;  // beyond the fixed scratch

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return RR_ERR_CUDA;
  }
  DevInfo d;  // attribute queries only: nothing here allocates
  d.device = dev;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cluster_launch, cudaDevAttrClusterLaunch, dev) != cudaSuccess) {
    cudaGetLastError();
    return RR_ERR_CUDA;
  }
  if (cluster_size > 1 && !d.cluster_launch) return RR_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> run(g_noalloc_run_mu);
  unsigned char *base = nullptr;
  int st = scratch_address(dev, &base);
  if (st != RR_OK) return st;
  void *vals = base;
  void *res = base + (size_t)kNoAllocMaxValues * 4;
  int64_t *counter = reinterpret_cast<int64_t *>(base + 2 * (size_t)kNoAllocMaxValues * 4);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Once anything is queued, every return waits for the stream first: work
  // left in flight on the shared array (say a fill whose all-reduce launch
  // was then refused) would otherwise overwrite the next caller's values
  // after the lock is released.
  auto finish = [&](int status) {
    if (cudaStreamSynchronize(s) != cudaSuccess && status == RR_OK) status = RR_ERR_CUDA;
    cudaGetLastError();
    return status;
  };
  // the array keeps the previous call's contents: the counter must restart at 0
  if (cudaMemsetAsync(counter, 0, sizeof(int64_t), s) != cudaSuccess) return finish(RR_ERR_CUDA);
  st = launch_fill_selftest_values(vals, n, dtype, seed, s);
  if (st == RR_OK)
    st = launch_cluster_allreduce(vals, clusters, cluster_size, width, op, dtype, iters,
                                  two_slot ? 1 : 0, 2000, res, counter, s, d);
  if (st != RR_OK) return finish(st);
  int64_t h = -1;
  if (cudaMemcpyAsync(&h, counter, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (vals_host &&
       cudaMemcpyAsync(vals_host, vals, (size_t)n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      (res_host &&
       cudaMemcpyAsync(res_host, res, (size_t)n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess))
    return finish(RR_ERR_CUDA);
  st = finish(RR_OK);
  if (st != RR_OK) return st;
  *mismatches_out = h;
  return h == 0 ? RR_OK : RR_ERR_MISMATCH;
}
