// reduce.cu -- row-wise monoid reduction in four tiers (the "reduce" page,
// algorithm/gpu/rowwise, tier semantics): warp, tiled/serial, block and
// split-K.  The split-K tier spreads one row over the CTAs of a thread-block
// cluster and combines the CTA partials with cluster_allreduce (the
// "cluster_allreduce" page).
//
// Every tier folds each row in a fixed order that depends only on the shape,
// the tier's compile-time geometry and the row's address alignment, so the
// same call gives the same bits on every run.
#include <climits>
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

// Geometry of the tiers (each can be overridden at build time).
#ifndef RR_BLOCK_THREADS
#define RR_BLOCK_THREADS 256
#endif
#ifndef RR_BLOCK_UNROLL
#define RR_BLOCK_UNROLL 8
#endif
#ifndef RR_WARP_UNROLL
#define RR_WARP_UNROLL 8
#endif
#ifndef RR_TILED_VECS
#define RR_TILED_VECS 8
#endif
#ifndef RR_TILED_UNROLL_MAX
#define RR_TILED_UNROLL_MAX 4
#endif
#ifndef RR_GRID_CAP
#define RR_GRID_CAP 1
#endif
#ifndef RR_TILED_MAX_NV
#define RR_TILED_MAX_NV 8
#endif

constexpr int kBlockThreads = RR_BLOCK_THREADS, kBlockUnroll = RR_BLOCK_UNROLL;
// Block tier on long rows: a CTA per row keeps threads x unroll 16-byte
// loads in flight, and with few rows per SM 256 x 8 is too little to cover
// HBM latency (152 rows of 441505 fp32: 2941 GB/s).  Rows of at least
// RR_BLOCK_LONG_COLS elements take 16 loads per thread (such a row spans two
// or more passes of them, so the predicated remainder stays small; shorter
// rows keep 8, which leaves room for more CTAs per SM).
#ifndef RR_BLOCK_LONG_COLS
#define RR_BLOCK_LONG_COLS 32768
#endif
constexpr int kBlockLongUnroll = 16;
constexpr int kSplitThreads = 512, kSplitUnroll = 8;
constexpr int kWarpBlock = 256, kWarpUnroll = RR_WARP_UNROLL;
constexpr int kTiledBlock = 256;
// Tiled tier: groups of rows each thread keeps in flight, so that a thread
// holds about RR_TILED_VECS vectors (NV vectors per row, EWT rows per group).
__host__ __device__ constexpr int tiled_unroll(int nv, int ewt) {
  // 8-float rows, a row a thread: 8 rows in flight a thread (with 4 CTAs an
  // SM, 64 registers); measured max / min 0.83 -> 0.86 of the copy
  // bandwidth back to back, sum unchanged (0.87), where wider rows lost
  return (nv == 2 && ewt == 1) ? 8 :
         RR_TILED_VECS / (nv * ewt) < 1
             ? 1
             : (RR_TILED_VECS / (nv * ewt) > RR_TILED_UNROLL_MAX ? RR_TILED_UNROLL_MAX
                                                                : RR_TILED_VECS / (nv * ewt));
}

// ---------------------------------------------------------------------------
// Fold elements [begin, end) of one row, as one thread of a THREADS-wide CTA.
// Scalar head up to the first 16-byte boundary, 128-bit streaming loads over
// the aligned body (UNROLL independent loads and accumulators per thread per
// step, so UNROLL * 16 bytes are in flight per thread), scalar tail.  The
// block tier folds whole rows with it; the split-K tier folds one slice.
// Returns this thread's partial (to be combined by block_reduce).
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int UNROLL>
__device__ __forceinline__ typename Op::T fold_range(const typename Op::T *__restrict__ p,
                                                     int64_t begin, int64_t end) {
  using T = typename Op::T;
  using V = typename Vec4<T>::type;
  const int tid = threadIdx.x;
  T acc[UNROLL];
#pragma unroll
  for (int u = 0; u < UNROLL; ++u) acc[u] = Op::id();
  const int64_t n = end - begin;
  if (n > 0) {
    const T *s = p + begin;
    int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)s & 15u)) & 15u) / sizeof(T));
    if (head > n) head = n;
    if (tid < head) acc[0] = Op::f(acc[0], __ldg(s + tid));
    const V *q = reinterpret_cast<const V *>(s + head);
    const int64_t nv = (n - head) >> 2;
    int64_t i = tid;
    for (; i + (int64_t)(UNROLL - 1) * THREADS < nv; i += (int64_t)UNROLL * THREADS) {
      V v[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) v[u] = ld_stream(q + i + (int64_t)u * THREADS);
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) acc[u] = fold4<Op>(acc[u], v[u]);
    }
#pragma unroll
    for (int u = 0; u < UNROLL - 1; ++u) {
      const int64_t k = i + (int64_t)u * THREADS;
      if (k < nv) acc[u] = fold4<Op>(acc[u], ld_stream(q + k));
    }
    const int64_t t0 = head + (nv << 2);
    if (tid < n - t0) acc[UNROLL - 1] = Op::f(acc[UNROLL - 1], __ldg(s + t0 + tid));
  }
  T a = acc[0];
#pragma unroll
  for (int u = 1; u < UNROLL; ++u) a = Op::f(a, acc[u]);
  return a;
}

// ---------------------------------------------------------------------------
// Block tier: one CTA per row, persistent grid-stride over rows.
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS)
k_block(const typename Op::T *__restrict__ x, int64_t rows, int64_t cols,
        typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  __shared__ T red[THREADS / 32];
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    T a = fold_range<Op, THREADS, UNROLL>(x + row * cols, 0, cols);
    a = block_reduce<Op, THREADS>(a, red);
    if (threadIdx.x == 0) out[row] = Op::finalize(a);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Warp tier, vector form: cols = 4 * LPR with LPR in {1, 2, 4, 8} and a
// 16-byte aligned base.  A warp covers 32 / LPR rows per 512-byte load (a
// segment of LPR lanes per row, one 128-bit vector per lane), folds the
// vector serially, then combines the segment with an xor butterfly of
// log2(LPR) steps.  U independent loads per lane are in flight.
// ---------------------------------------------------------------------------
template <class Op, int LPR, int U>
__global__ void __launch_bounds__(kWarpBlock)
k_warp_vec(const typename Op::T *__restrict__ x, int64_t rows,
           typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  using V = typename Vec4<T>::type;
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31, seg = lane / LPR, sub = lane % LPR;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const V *q = reinterpret_cast<const V *>(x);
  for (int64_t r0 = warp * (RPW * U); r0 < rows; r0 += nwarps * (RPW * U)) {
    // Unconditional loads (a row past the end re-reads the last row, a valid
    // address; its value is dropped below), so all U go out back to back.
    V v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = r0 + u * RPW + seg;
      v[u] = ld_stream(q + (row < rows ? row : rows - 1) * LPR + sub);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = r0 + u * RPW + seg;
      T a = row < rows ? fold4<Op>(Op::id(), v[u]) : Op::id();
      a = warp_allreduce<Op, LPR>(a);
      if (sub == 0 && row < rows) out[row] = Op::finalize(a);
    }
  }
}

// Warp tier, scalar form (the page's literal reading): lane i loads element
// i of the row (any alignment, cols <= 32), then a 5-step xor butterfly.
template <class Op, int U>
__global__ void __launch_bounds__(kWarpBlock)
k_warp_scalar(const typename Op::T *__restrict__ x, int64_t rows, int cols,
              typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r0 = warp * U; r0 < rows; r0 += nwarps * U) {
    T v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = r0 + u;
      v[u] = (row < rows && lane < cols) ? __ldg(x + row * cols + lane) : Op::id();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const T a = warp_allreduce<Op, 32>(v[u]);
      if (lane == 0 && r0 + u < rows) out[r0 + u] = Op::finalize(a);
    }
  }
}

// ---------------------------------------------------------------------------
// Warp tier for rows longer than a warp ("reduce" page, warp tier, read for
// rows wider than 32: the lanes of a warp segment stride the row).  A
// segment of LPR lanes owns a row; lane `sub` folds units sub, sub + LPR, ...
// of it (VEC: 16-byte vectors, else single elements), KV per pass: the KV
// loads go out first and are folded last-loaded first, so the first fold
// needs the last load and all KV are in flight together (a unit past the
// row's end re-reads the row's last unit and is not folded); passes repeat
// until the row is covered; then an xor butterfly over the segment.  32 / LPR rows per warp,
// grid-stride over warps; no shared memory and no barrier, so rows of 33 to
// a few thousand elements need no 256-thread CTA each.
// ---------------------------------------------------------------------------
template <class Op, bool VEC, int LPR, int KV>
__global__ void __launch_bounds__(kWarpBlock)
k_warp_seg(const typename Op::T *__restrict__ x, int64_t rows, int64_t cols,
           typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  using V = typename Vec4<T>::type;
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31, seg = lane / LPR, sub = lane % LPR;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n = VEC ? cols / 4 : cols;  // units per row
  for (int64_t r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
    const int64_t row = r0 + seg;
    // a segment past the last row re-reads the last row and writes nothing
    const int64_t rr = row < rows ? row : rows - 1;
    T acc = Op::id();
    for (int64_t k0 = sub; k0 < n; k0 += (int64_t)KV * LPR) {
      if constexpr (VEC) {
        const V *q = reinterpret_cast<const V *>(x) + rr * n;
        V v[KV];
#pragma unroll
        for (int j = 0; j < KV; ++j) {
          const int64_t k = k0 + (int64_t)j * LPR;
          v[j] = ld_stream(q + (k < n ? k : n - 1));
        }
#pragma unroll
        for (int j = KV - 1; j >= 0; --j)
          if (k0 + (int64_t)j * LPR < n) acc = fold4<Op>(acc, v[j]);
      } else {
        const T *q = x + rr * n;
        T v[KV];
#pragma unroll
        for (int j = 0; j < KV; ++j) {
          const int64_t k = k0 + (int64_t)j * LPR;
          v[j] = __ldg(q + (k < n ? k : n - 1));
        }
#pragma unroll
        for (int j = KV - 1; j >= 0; --j)
          if (k0 + (int64_t)j * LPR < n) acc = Op::f(acc, v[j]);
      }
    }
    acc = warp_allreduce<Op, LPR>(acc);
    if (sub == 0 && row < rows) out[row] = Op::finalize(acc);
  }
}

// ---------------------------------------------------------------------------
// Tiled tier: a thread owns EWT adjacent rows and folds them on its own (no
// cross-thread combine).  Vector form: cols = 4 * NV, 16-byte aligned base;
// with V8 (NV even, 32-byte aligned base) each row is read with 256-bit
// loads, so a warp instruction covers 32 * 32 contiguous bytes.
// ---------------------------------------------------------------------------
template <class Op, int NV, int EWT, bool V8, int U>
// Narrow rows (NV * EWT <= 2): held to 32 registers, 8 CTAs per SM, so the
// persistent grid covers the usual row counts in one pass of loads per
// thread (the max / min forms otherwise took 40 and a second pass).
#ifndef RR_TILED_MIN_BLOCKS
#define RR_TILED_MIN_BLOCKS 8
#endif
__global__ void __launch_bounds__(kTiledBlock, (NV == 2 && EWT == 1) ? 4 : ((NV * EWT <= 2) ? RR_TILED_MIN_BLOCKS : 1))
k_tiled_vec(const typename Op::T *__restrict__ x, int64_t rows,
            typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  using V = typename Vec4<T>::type;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  const int64_t groups = (rows + EWT - 1) / EWT;
  const V *q = reinterpret_cast<const V *>(x);
  for (int64_t g0 = tid; g0 < groups; g0 += nth * U) {
    V v[U][EWT][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + (int64_t)u * nth;
#pragma unroll
      for (int e = 0; e < EWT; ++e) {
        // unconditional loads: a row past the end re-reads the last row (a
        // valid address) and is dropped below, so all loads go out back to back
        const int64_t row = g * EWT + e;
        const int64_t rl = row < rows ? row : rows - 1;
        if (V8) {
#pragma unroll
          for (int k = 0; k < NV; k += 2) {
            uint32_t r8[8];
            ld_stream_v8(q + rl * NV + k, r8);
            v[u][e][k].x = from_bits<T>(r8[0]); v[u][e][k].y = from_bits<T>(r8[1]);
            v[u][e][k].z = from_bits<T>(r8[2]); v[u][e][k].w = from_bits<T>(r8[3]);
            v[u][e][k + 1].x = from_bits<T>(r8[4]); v[u][e][k + 1].y = from_bits<T>(r8[5]);
            v[u][e][k + 1].z = from_bits<T>(r8[6]); v[u][e][k + 1].w = from_bits<T>(r8[7]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < NV; ++k) v[u][e][k] = ld_stream(q + rl * NV + k);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + (int64_t)u * nth;
#pragma unroll
      for (int e = 0; e < EWT; ++e) {
        const int64_t row = g * EWT + e;
        T a = Op::id();
#pragma unroll
        for (int k = 0; k < NV; ++k) a = fold4<Op>(a, v[u][e][k]);
        if (g < groups && row < rows) out[row] = Op::finalize(a);
      }
    }
  }
}

// Tiled / serial tier, scalar form: any cols, any alignment; a thread folds
// its EWT rows element by element.
template <class Op, int EWT>
__global__ void __launch_bounds__(kTiledBlock)
k_tiled_scalar(const typename Op::T *__restrict__ x, int64_t rows, int64_t cols,
               typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  const int64_t groups = (rows + EWT - 1) / EWT;
  for (int64_t g = tid; g < groups; g += nth) {
#pragma unroll
    for (int e = 0; e < EWT; ++e) {
      const int64_t row = g * EWT + e;
      if (row < rows) {
        T a = Op::id();
        const T *p = x + row * cols;
        for (int64_t i = 0; i < cols; ++i) a = Op::f(a, __ldg(p + i));
        out[row] = Op::finalize(a);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Split-K tier ("reduce" page, split-K tier; "cluster_allreduce" page).
// A cluster of C CTAs per row; CTA rank r folds slice r of the row.  Slices
// are ceil(cols / C) elements rounded up to a multiple of 4 and shifted down
// by the row's misalignment, so every slice but the first starts on a
// 16-byte boundary; the last slice takes the remainder.  The CTA partials
// are combined with cluster_allreduce: every CTA gathers every peer and
// folds in rank order, so all C copies of the result are bit-identical.
// Rank 0 writes out[row]; rank_out (optional) receives every rank's copy.
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS)
k_splitk(const typename Op::T *__restrict__ x, int64_t rows, int64_t cols,
         typename Op::T *__restrict__ out, typename Op::T *__restrict__ rank_out) {
  pdl_begin();
  using T = typename Op::T;
  __shared__ T red[THREADS / 32];
  __shared__ T slot[2];
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t row = cluster_id_x();
  const T *p = x + row * cols;
  const int64_t chunk = ((cols + C - 1) / C + 3) & ~int64_t(3);
  const int64_t mis = (int64_t)(((uint32_t)(uintptr_t)p & 15u) / sizeof(T));
  auto bound = [&](int64_t k) -> int64_t {
    if (k == 0) return 0;
    if (k >= (int64_t)C) return cols;
    const int64_t b = k * chunk - mis;
    return b < 0 ? 0 : (b > cols ? cols : b);
  };
  T a = fold_range<Op, THREADS, UNROLL>(p, bound(r), bound(r + 1));
  a = block_reduce<Op, THREADS>(a, red);
  const T v[1] = {a};
  T res[1];
  cluster_allreduce<Op, 1>(slot, v, C, /*tail_sync=*/true, res);
  if (threadIdx.x == 0) {
    const T fin = Op::finalize(res[0]);
    if (r == 0) out[row] = fin;
    if (rank_out) rank_out[row * C + r] = fin;
  }
}

// ---------------------------------------------------------------------------
// Multi-cluster split-K: G clusters of C CTAs per row, for rows too few to
// cover the GPU with one cluster each.  The row is cut into G*C slices (as
// the split-K tier cuts it into C); cluster g of the row folds slices
// g*C .. g*C + C - 1, combines its CTAs with cluster_allreduce and rank 0
// stores the cluster's partial in partial[row * G + g].  A second kernel
// folds the G partials of each row in order g = 0..G-1.  Every step has a
// fixed order, so the result is the same on every run.
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int UNROLL>
__global__ void __launch_bounds__(THREADS)
k_splitk_multi(const typename Op::T *__restrict__ x, int64_t rows, int64_t cols, int G,
               typename Op::T *__restrict__ partial) {
  pdl_begin();
  using T = typename Op::T;
  __shared__ T red[THREADS / 32];
  __shared__ T slot[2];
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t cid = cluster_id_x();
  const int64_t row = cid / G, g = cid - row * G;
  const T *p = x + row * cols;
  const int64_t S = (int64_t)G * C;
  const int64_t chunk = ((cols + S - 1) / S + 3) & ~int64_t(3);
  const int64_t mis = (int64_t)(((uint32_t)(uintptr_t)p & 15u) / sizeof(T));
  auto bound = [&](int64_t k) -> int64_t {
    if (k == 0) return 0;
    if (k >= S) return cols;
    const int64_t b = k * chunk - mis;
    return b < 0 ? 0 : (b > cols ? cols : b);
  };
  const int64_t k0 = g * C + r;
  T a = fold_range<Op, THREADS, UNROLL>(p, bound(k0), bound(k0 + 1));
  a = block_reduce<Op, THREADS>(a, red);
  const T v[1] = {a};
  T res[1];
  cluster_allreduce<Op, 1>(slot, v, C, /*tail_sync=*/true, res);
  if (r == 0 && threadIdx.x == 0) partial[row * G + g] = res[0];
}

template <class Op>
__global__ void k_fold_partials(const typename Op::T *__restrict__ partial, int64_t rows, int G,
                                typename Op::T *__restrict__ out) {
  pdl_begin();
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  typename Op::T acc = partial[row * G];
  for (int g = 1; g < G; ++g) acc = Op::f(acc, partial[row * G + g]);
  out[row] = Op::finalize(acc);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
template <class K>
int grid_for(K kernel, int threads, int64_t work_blocks, const DevInfo &d, int smem = 0) {
  int64_t g = work_blocks;
  if (RR_GRID_CAP) {  // persistent: at most one wave of resident CTAs
    const int nb = occupancy_blocks((const void *)kernel, threads, (size_t)smem, d.device);
    const int64_t cap = (int64_t)nb * d.sm_count;
    if (g > cap) g = cap;
  }
  if (g > 0x7fffffffLL) g = 0x7fffffffLL;
  return (int)(g < 1 ? 1 : g);
}

template <class Op>
int launch_splitk_kernel(const void *x, int64_t rows, int64_t cols, void *out,
                         void *rank_out, int C, cudaStream_t s) {
  using T = typename Op::T;
  auto kern = k_splitk<Op, kSplitThreads, kSplitUnroll>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return cuda_status(launch_kernel(kern, dim3((unsigned)(rows * C)), dim3(kSplitThreads), 0, s, C,
                                   (const T *)x, rows, cols, (T *)out, (T *)rank_out));
}

template <class Op>
int max_cluster_for(int want, const DevInfo &d) {
  auto kern = k_splitk<Op, kSplitThreads, kSplitUnroll>;
  for (int C = 16; C >= 1; C >>= 1) {
    if (C > want) continue;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (C == 1) return 1;
    if (occupancy_clusters((const void *)kern, kSplitThreads, 0, C, d.device) > 0) return C;
  }
  return 0;
}

template <class Op>
int launch_tier(const void *xv, int64_t rows, int64_t cols, void *outv, cudaStream_t s,
                int tier, int C, int ewt, void *rank_out, const DevInfo &d) {
  using T = typename Op::T;
  const T *x = (const T *)xv;
  T *out = (T *)outv;
  const uintptr_t a = (uintptr_t)xv;
  switch (tier) {
    case RR_TIER_BLOCK: {
      if (cols >= RR_BLOCK_LONG_COLS) {
        auto k = k_block<Op, kBlockThreads, kBlockLongUnroll>;
        const int g = grid_for(k, kBlockThreads, rows, d);
        launch_kernel(k, dim3(g), dim3(kBlockThreads), 0, s, 0, x, rows, cols, out);
        return cuda_status(cudaGetLastError());
      }
      auto k = k_block<Op, kBlockThreads, kBlockUnroll>;
      const int g = grid_for(k, kBlockThreads, rows, d);
      launch_kernel(k, dim3(g), dim3(kBlockThreads), 0, s, 0, x, rows, cols, out);
      return cuda_status(cudaGetLastError());
    }
    case RR_TIER_WARP: {
      if (cols > 32) {
        // a segment of LPR lanes per row, 8 units per lane and pass, at least
        // 32 bytes per segment and pass (2 vector lanes, 8 scalar lanes), at
        // most 32: enough lanes to cover the row in one pass (long rows then
        // read 32 lanes' worth of contiguous bytes per instruction), halved
        // while more than 30% of the slots would fall past the row's end
        const bool vec = (cols % 4 == 0) && (a % 16 == 0);
        const int64_t n = vec ? cols / 4 : cols;
        const int lmin = vec ? 2 : 8;
        auto fill = [n](int l) {
          const int64_t per = (int64_t)l * 8;
          return (double)n / (double)((n + per - 1) / per * per);
        };
        int lpr = lmin;
        while (lpr < 32 && (int64_t)lpr * 8 < n) lpr *= 2;
        while (lpr > lmin && fill(lpr) < 0.7 && fill(lpr / 2) > fill(lpr)) lpr /= 2;
        const int64_t rows_per_block = (int64_t)(kWarpBlock / 32) * (32 / lpr);
        const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
#define RR_WARP_SEG(VEC, L)                                                    \
  {                                                                            \
    auto k = k_warp_seg<Op, VEC, L, 8>;                                        \
    const int g = grid_for(k, kWarpBlock, blocks, d);                          \
    launch_kernel(k, dim3(g), dim3(kWarpBlock), 0, s, 0, x, rows, cols, out);  \
    break;                                                                     \
  }
        if (vec) {
          switch (lpr) {
            case 2: RR_WARP_SEG(true, 2)
            case 4: RR_WARP_SEG(true, 4)
            case 8: RR_WARP_SEG(true, 8)
            case 16: RR_WARP_SEG(true, 16)
            default: RR_WARP_SEG(true, 32)
          }
        } else {
          switch (lpr) {
            case 8: RR_WARP_SEG(false, 8)
            case 16: RR_WARP_SEG(false, 16)
            default: RR_WARP_SEG(false, 32)
          }
        }
#undef RR_WARP_SEG
        return cuda_status(cudaGetLastError());
      }
      const bool vec = (cols % 4 == 0) && cols >= 4 && (a % 16 == 0) &&
                       (cols == 4 || cols == 8 || cols == 16 || cols == 32);
      if (vec) {
        const int lpr = (int)(cols / 4);
        const int64_t rows_per_block = (int64_t)(kWarpBlock / 32) * (32 / lpr) * kWarpUnroll;
        const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
#define RR_WARP_VEC(L)                                                         \
  {                                                                            \
    auto k = k_warp_vec<Op, L, kWarpUnroll>;                                   \
    const int g = grid_for(k, kWarpBlock, blocks, d);                          \
    launch_kernel(k, dim3(g), dim3(kWarpBlock), 0, s, 0, x, rows, out);                                  \
    break;                                                                     \
  }
        switch (lpr) {
          case 1: RR_WARP_VEC(1)
          case 2: RR_WARP_VEC(2)
          case 4: RR_WARP_VEC(4)
          default: RR_WARP_VEC(8)
        }
#undef RR_WARP_VEC
      } else {
        auto k = k_warp_scalar<Op, kWarpUnroll>;
        const int64_t rows_per_block = (int64_t)(kWarpBlock / 32) * kWarpUnroll;
        const int g = grid_for(k, kWarpBlock, (rows + rows_per_block - 1) / rows_per_block, d);
        launch_kernel(k, dim3(g), dim3(kWarpBlock), 0, s, 0, x, rows, (int)cols, out);
      }
      return cuda_status(cudaGetLastError());
    }
    case RR_TIER_TILED: {
      const int e = (ewt == 2 || ewt == 4) ? ewt : 1;
      const int64_t groups = (rows + e - 1) / e;
      // rows of up to 8 vectors; 5 to 8 only with a row per thread
      const bool vec = cols >= 4 && cols <= 4 * RR_TILED_MAX_NV && cols % 4 == 0 &&
                       (a % 16 == 0) && (cols <= 16 || e == 1);
      if (vec) {
        const int nv = (int)(cols / 4);
        const bool v8 = (nv % 2 == 0) && (a % 32 == 0);
        const int64_t blocks = (groups + kTiledBlock - 1) / kTiledBlock;
#define RR_TILED_VEC(NV, E, V8)                                                \
  {                                                                            \
    auto k = k_tiled_vec<Op, NV, E, V8, tiled_unroll(NV, E)>;                  \
    const int g = grid_for(k, kTiledBlock, blocks, d);                         \
    launch_kernel(k, dim3(g), dim3(kTiledBlock), 0, s, 0, x, rows, out);                                 \
  }
#define RR_TILED_E(NV, V8)                                                     \
  {                                                                            \
    if (e == 1) RR_TILED_VEC(NV, 1, V8)                                        \
    else if (e == 2) RR_TILED_VEC(NV, 2, V8)                                   \
    else RR_TILED_VEC(NV, 4, V8)                                               \
  }
        if (nv == 1) RR_TILED_E(1, false)
        else if (nv == 2) { if (v8) RR_TILED_E(2, true) else RR_TILED_E(2, false) }
        else if (nv == 3) RR_TILED_E(3, false)
        else if (nv == 4) { if (v8) RR_TILED_E(4, true) else RR_TILED_E(4, false) }
#if RR_TILED_MAX_NV > 4
        else if (nv == 5) RR_TILED_VEC(5, 1, false)
        else if (nv == 6) { if (v8) RR_TILED_VEC(6, 1, true) else RR_TILED_VEC(6, 1, false) }
        else if (nv == 7) RR_TILED_VEC(7, 1, false)
        else { if (v8) RR_TILED_VEC(8, 1, true) else RR_TILED_VEC(8, 1, false) }
#endif
#undef RR_TILED_E
#undef RR_TILED_VEC
      } else {
        const int64_t blocks = (groups + kTiledBlock - 1) / kTiledBlock;
        if (e == 1) {
          auto k = k_tiled_scalar<Op, 1>;
          launch_kernel(k, dim3(grid_for(k, kTiledBlock, blocks, d)), dim3(kTiledBlock), 0, s, 0, x, rows, cols, out);
        } else if (e == 2) {
          auto k = k_tiled_scalar<Op, 2>;
          launch_kernel(k, dim3(grid_for(k, kTiledBlock, blocks, d)), dim3(kTiledBlock), 0, s, 0, x, rows, cols, out);
        } else {
          auto k = k_tiled_scalar<Op, 4>;
          launch_kernel(k, dim3(grid_for(k, kTiledBlock, blocks, d)), dim3(kTiledBlock), 0, s, 0, x, rows, cols, out);
        }
      }
      return cuda_status(cudaGetLastError());
    }
    case RR_TIER_SPLITK:
      return launch_splitk_kernel<Op>(xv, rows, cols, outv, rank_out, C, s);
    default:
      return RR_ERR_INVALID;
  }
}

template <class Op>
int launch_splitk_multi(const void *x, int64_t rows, int64_t cols, void *out, int C, int G,
                        void *ws, cudaStream_t s) {
  using T = typename Op::T;
  auto kern = k_splitk_multi<Op, kSplitThreads, kSplitUnroll>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (log_enabled())
    std::fprintf(stderr, "rr: reduce split-K multi rows=%lld cols=%lld C=%d G=%d\n",
                 (long long)rows, (long long)cols, C, G);
  cudaError_t e = launch_kernel(kern, dim3((unsigned)(rows * G * C)), dim3(kSplitThreads), 0, s, C,
                                (const T *)x, rows, cols, G, (T *)ws);
  if (e != cudaSuccess) return cuda_status(e);
  launch_kernel(k_fold_partials<Op>, dim3((unsigned)((rows + 255) / 256)), dim3(256), 0, s, 0, (const T *)ws, rows, G,
                                                                     (T *)out);
  return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_reduce_splitk_multi(const void *x, int64_t rows, int64_t cols, int op, int dtype,
                               void *out, int C, int G, void *ws, cudaStream_t s) {
  if (dtype == RR_F32) {
    if (op == RR_OP_SUM) return launch_splitk_multi<SumF32>(x, rows, cols, out, C, G, ws, s);
    if (op == RR_OP_MAX) return launch_splitk_multi<MaxF32>(x, rows, cols, out, C, G, ws, s);
    return launch_splitk_multi<MinF32>(x, rows, cols, out, C, G, ws, s);
  }
  if (op == RR_OP_SUM) return launch_splitk_multi<SumI32>(x, rows, cols, out, C, G, ws, s);
  if (op == RR_OP_MAX) return launch_splitk_multi<MaxI32>(x, rows, cols, out, C, G, ws, s);
  return launch_splitk_multi<MinI32>(x, rows, cols, out, C, G, ws, s);
}

int splitk_max_cluster(int op, int dtype, int want, const DevInfo &d) {
  (void)d;
  if (dtype == RR_F32) {
    if (op == RR_OP_SUM) return max_cluster_for<SumF32>(want, d);
    if (op == RR_OP_MAX) return max_cluster_for<MaxF32>(want, d);
    return max_cluster_for<MinF32>(want, d);
  }
  if (op == RR_OP_SUM) return max_cluster_for<SumI32>(want, d);
  if (op == RR_OP_MAX) return max_cluster_for<MaxI32>(want, d);
  return max_cluster_for<MinI32>(want, d);
}

int launch_reduce(const void *x, int64_t rows, int64_t cols, int op, int dtype, void *out,
                  cudaStream_t s, int tier, int C, int ewt, void *rank_out, const DevInfo &d) {
  if (dtype == RR_F32) {
    if (op == RR_OP_SUM) return launch_tier<SumF32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
    if (op == RR_OP_MAX) return launch_tier<MaxF32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
    return launch_tier<MinF32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
  }
  if (op == RR_OP_SUM) return launch_tier<SumI32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
  if (op == RR_OP_MAX) return launch_tier<MaxI32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
  return launch_tier<MinI32>(x, rows, cols, out, s, tier, C, ewt, rank_out, d);
}

}  // namespace rr
