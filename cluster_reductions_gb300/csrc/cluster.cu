// cluster.cu -- the cluster all-reduce primitive (the "cluster_allreduce"
// page) run back to back by several clusters, with a per-thread bit check
// against the rank-order fold; the seeded value generator of its self-test;
// and the bounded-wait probe used to test failure detection.
#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

constexpr int kCaThreads = 128;

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// Iteration t, cluster cl, rank r reads vals[((t*ncl + cl)*C + r)*W + j].
// Only thread 0 loads an input; the other threads start from the identity
// ("cluster_allreduce" page, arguments: the per-CTA vector is the result of
// a block reduction, so only its copy in thread 0 counts).  With skew > 0, thread 0 of each rank first
// spins (hash & 7) * skew clock cycles, so ranks arrive out of step.
template <class Op, int W>
__global__ void __launch_bounds__(kCaThreads)
k_cluster_allreduce(const typename Op::T *__restrict__ vals, typename Op::T *__restrict__ res,
                    int iters, int two_slot, int64_t skew,
                    unsigned long long *__restrict__ mismatches) {
  pdl_begin();
  using T = typename Op::T;
  __shared__ T slot[2][2 * W];
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const uint32_t cl = cluster_id_x(), ncl = cluster_nid_x();
  unsigned long long bad = 0;
  for (int t = 0; t < iters; ++t) {
    const int64_t base = ((int64_t)t * ncl + cl) * C * W;
    const T *vin = vals + base;
    T v[W];
#pragma unroll
    for (int j = 0; j < W; ++j) v[j] = (threadIdx.x == 0) ? vin[r * W + j] : Op::id();
    if (skew > 0 && threadIdx.x == 0) {
      const uint64_t h = splitmix64(((uint64_t)t << 32) ^ ((uint64_t)cl << 8) ^ r);
      const int64_t delay = (int64_t)(h & 7u) * skew;
      const long long t0 = clock64();
      while (clock64() - t0 < delay) {
      }
    }
    T o[W];
    cluster_allreduce<Op, W>(two_slot ? slot[t & 1] : slot[0], v, C, two_slot == 0, o);
    if (threadIdx.x == 0) {
#pragma unroll
      for (int j = 0; j < W; ++j) res[base + r * W + j] = o[j];
    }
    if (mismatches) {  // without a counter the kernel only times the combines
#pragma unroll
      for (int j = 0; j < W; ++j) {
        T e = __ldg(vin + j);
        for (uint32_t q = 1; q < C; ++q) e = Op::f(e, __ldg(vin + q * W + j));
        if (to_bits<T>(e) != to_bits<T>(o[j])) ++bad;
      }
    }
  }
  // Without the per-combine tail sync a CTA must not exit while a peer may
  // still read its last slot.
  if (two_slot && C > 1) cluster_sync();
  if (bad && mismatches) atomicAdd(mismatches, bad);
}

// Seeded per-rank values: fp32 with widely spread magnitudes (so the fold
// order shows in the bits), or full-range int32 (so sums wrap).
__global__ void k_fill(void *vals, int64_t n, int dtype, uint64_t seed) {
  pdl_begin();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t u = splitmix64(seed ^ splitmix64((uint64_t)i));
    if (dtype == RR_F32) {
      const float mant = (float)(u >> 40) * (1.0f / 16777216.0f) * 2.0f - 1.0f;
      const int ex = (int)((u >> 8) % 41u) - 20;
      ((float *)vals)[i] = ldexpf(mant, ex);
    } else {
      ((int *)vals)[i] = (int)(uint32_t)(u >> 32);
    }
  }
}

// Failure-detection probe: an mbarrier expecting two arrivals gets one, so
// its phase never completes; the bounded wait gives up and records
// kErrTimeout.  Nothing is in flight, so the kernel then returns normally.
__global__ void k_wait_probe(int64_t budget, int *err) {
  pdl_begin();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bar);
    if (!mbar_wait_bounded(&bar, 0, budget)) set_error(err, kErrTimeout);
  }
}

template <class Op, int W>
int launch_ca_w(const void *vals, int clusters, int C, int iters, int two_slot, int64_t skew,
                void *res, int64_t *mism, cudaStream_t s, int device) {
  using T = typename Op::T;
  auto kern = k_cluster_allreduce<Op, W>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  // Clusters do not wait on one another, so one co-resident cluster
  // (n >= 1) suffices.
  if (C > 1 && occupancy_clusters((const void *)kern, kCaThreads, 0, C, device) < 1)
    return RR_ERR_UNSUPPORTED;
  return cuda_status(launch_kernel(kern, dim3((unsigned)(clusters * C)), dim3(kCaThreads), 0, s, C,
                                   (const T *)vals, (T *)res, iters, two_slot, skew,
                                   (unsigned long long *)mism));
}

template <class Op>
int launch_ca(const void *vals, int clusters, int C, int W, int iters, int two_slot,
              int64_t skew, void *res, int64_t *mism, cudaStream_t s, int dev) {
  switch (W) {
    case 1: return launch_ca_w<Op, 1>(vals, clusters, C, iters, two_slot, skew, res, mism, s, dev);
    case 2: return launch_ca_w<Op, 2>(vals, clusters, C, iters, two_slot, skew, res, mism, s, dev);
    case 4: return launch_ca_w<Op, 4>(vals, clusters, C, iters, two_slot, skew, res, mism, s, dev);
    case 8: return launch_ca_w<Op, 8>(vals, clusters, C, iters, two_slot, skew, res, mism, s, dev);
    default: return RR_ERR_INVALID;
  }
}

}  // namespace

int launch_cluster_allreduce(const void *vals, int clusters, int C, int width, int op, int dtype,
                             int iters, int two_slot, int64_t skew_cycles, void *res,
                             int64_t *mismatches, cudaStream_t s, const DevInfo &d) {
  if (dtype == RR_F32) {
    if (op == RR_OP_SUM) return launch_ca<SumF32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
    if (op == RR_OP_MAX) return launch_ca<MaxF32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
    return launch_ca<MinF32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
  }
  if (op == RR_OP_SUM) return launch_ca<SumI32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
  if (op == RR_OP_MAX) return launch_ca<MaxI32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
  return launch_ca<MinI32>(vals, clusters, C, width, iters, two_slot, skew_cycles, res, mismatches, s, d.device);
}

int launch_fill_selftest_values(void *vals, int64_t n, int dtype, uint64_t seed, cudaStream_t s) {
  if (n <= 0) return RR_OK;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  launch_kernel(k_fill, dim3((unsigned)blocks), dim3(256), 0, s, 0, vals, n, dtype, seed);
  return cuda_status(cudaGetLastError());
}

int launch_wait_timeout_probe(int64_t budget, cudaStream_t s, const DevInfo &d) {
  launch_kernel(k_wait_probe, dim3(1), dim3(32), 0, s, 0, budget, d.err_word);
  return cuda_status(cudaGetLastError());
}

}  // namespace rr
