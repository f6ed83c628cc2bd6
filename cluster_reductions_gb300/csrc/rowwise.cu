// rowwise.cu -- the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise): softmax (pass 1 reduces the online-softmax
// (max, sum) monoid, pass 2 is a stateless map that writes exp(x - m) / s)
// and the layernorm statistics (mean, then the variance about the mean, both
// block reduces over the on-chip row).
//
// This file holds the block tier -- fast path: one CTA per row with the
// whole row held in registers, so the row is read from HBM exactly once;
// generic path (any width, any alignment): the row is streamed from global
// memory once per pass -- and the split-K tier (a cluster of CTAs per row,
// the slices read from global memory), and the tier choice (plan_rowwise).
// Many short rows take the warp tier (rowwarp.cu); long rows are staged in
// shared memory (rowstaged.cu).
#include <cstdio>

#include <cuda_bf16.h>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"
#include "rowwise.cuh"

namespace rr {
namespace {

#ifndef RR_ROW_THREADS
#define RR_ROW_THREADS 256
#endif
constexpr int kRowThreads = RR_ROW_THREADS;

// Block reduce of the (max, sum) pair; every thread receives the result.
template <int THREADS>
__device__ __forceinline__ void ms_block_allreduce(float &m, float &s, float *red_m,
                                                   float *red_s) {
  constexpr int NW = THREADS / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    ms_combine(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  if (lane == 0) { red_m[w] = m; red_s[w] = s; }
  __syncthreads();
  if (w == 0) {
    m = lane < NW ? red_m[lane] : -INFINITY;
    s = lane < NW ? red_s[lane] : 0.0f;
#pragma unroll
    for (int o = pow2_ceil(NW) / 2; o > 0; o >>= 1)
      ms_combine(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    if (lane == 0) { red_m[NW] = m; red_s[NW] = s; }
  }
  __syncthreads();
  m = red_m[NW];
  s = red_s[NW];
}

// Block sum returned to every thread with one barrier: an xor butterfly in
// each warp (every lane ends with the same bits), the warp sums to `red`, one
// barrier, then every thread folds red[0..NW-1] in warp order.  Consecutive
// calls must alternate between two `red` buffers: a thread may still be
// reading one call's sums while a faster thread writes the next call's, and
// the barrier of the call in between keeps the third call off the first
// buffer.  (The (max, sum) pair above keeps its two barriers: folding NW
// pairs in every thread costs more exp2 than the barrier saves.)
template <int THREADS>
__device__ __forceinline__ float sum_block_allreduce(float v, float *red) {
  constexpr int NW = THREADS / 32;
  v = warp_allreduce<SumF32, 32>(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) t += red[i];
  return t;
}

// ---------------------------------------------------------------------------
// Softmax, register-resident row.  Thread t holds vectors k*THREADS + t,
// k < NV, of the row (EPV elements each).  Pass 1: the thread's own (max,
// sum) over its elements, keeping p = e^(x - m_t) in registers; block
// (max, sum) reduce gives (M, S).  Pass 2: y = p * e^(m_t - M) / S, written
// with 32-byte streaming stores.  Requires cols % EPV == 0, x 16-byte and
// y 32-byte aligned (y 16-byte aligned for fp32 input).
// ---------------------------------------------------------------------------
template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_softmax_reg(const typename In::S *__restrict__ x, int64_t rows, int cols,
              float *__restrict__ y) {
  pdl_begin();
  constexpr int EPV = In::EPV;
  __shared__ float red_m[THREADS / 32 + 1], red_s[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  const int nvec = cols / EPV;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    using W = typename In::W;
    const W *q = reinterpret_cast<const W *>(x + row * (int64_t)cols);
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        In::unpack(In::ldv(q + idx), v[k]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = -INFINITY;
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < EPV; ++e) m = fmaxf(m, v[k][e]);
    float s = 0.0f;
    if (m != -INFINITY) {
      const float mb = m * kLog2e;
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float p = ex2_approx(fmaf(v[k][e], kLog2e, -mb));
          v[k][e] = p;
          s += p;
        }
    } else {
      // every element this thread holds is -inf: e^(x - M) = 0 (and not
      // -inf * 0 = NaN in the write below)
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
    }
    float M = m, S = s;
    ms_block_allreduce<THREADS>(M, S, red_m, red_s);
    const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S);
    float *yr = y + row * (int64_t)cols;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        if constexpr (EPV == 8) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = v[k][e % EPV] * f;
          st_stream_v8(yr + (int64_t)idx * EPV, o);
        } else if constexpr (EPV == 4) {
          st_stream_v4(yr + (int64_t)idx * EPV, v[k][0] * f, v[k][1 % EPV] * f,
                       v[k][2 % EPV] * f, v[k][3 % EPV] * f);
        } else {
          *reinterpret_cast<float2 *>(yr + (int64_t)idx * EPV) =
              make_float2(v[k][0] * f, v[k][1 % EPV] * f);
        }
      }
    }
    __syncthreads();
  }
}

// Softmax, generic: any cols, any alignment.  Pass 1 streams the row with an
// online (max, sum) update per element; pass 2 re-reads it and writes.
template <int THREADS, class In>
__global__ void __launch_bounds__(THREADS)
k_softmax_gen(const typename In::S *__restrict__ x, int64_t rows, int64_t cols,
              float *__restrict__ y) {
  pdl_begin();
  __shared__ float red_m[THREADS / 32 + 1], red_s[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const typename In::S *p = x + row * cols;
    float m = -INFINITY, s = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) ms_combine(m, s, In::load1(p + i), 1.0f);
    ms_block_allreduce<THREADS>(m, s, red_m, red_s);
    const float inv = 1.0f / s;
    const float mb = m * kLog2e;
    float *yr = y + row * cols;
    for (int64_t i = tid; i < cols; i += THREADS)
      yr[i] = (m == -INFINITY) ? 0.0f : ex2_approx(fmaf(In::load1(p + i), kLog2e, -mb)) * inv;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Layernorm statistics, register-resident row: mean = sum / cols (block
// sum), var = sum (x - mean)^2 / cols (second block sum over the registers),
// rstd = 1 / sqrt(var + eps).  Requires cols % EPV == 0 and x 16-byte aligned.
// The next row's raw vectors are loaded as soon as the current row is
// unpacked, so the loads stay in flight across the two block reductions.
// ---------------------------------------------------------------------------
template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_lnstats_reg(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
              float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  constexpr int EPV = In::EPV;
  __shared__ float red[2][THREADS / 32];
  const int tid = threadIdx.x;
  const int nvec = cols / EPV;
  const float inv_n = 1.0f / (float)cols;
  using W = typename In::W;
  W raw[NV];
  auto fetch = [&](int64_t r) {
    const W *q = reinterpret_cast<const W *>(x + r * (int64_t)cols);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) raw[k] = In::ldv(q + idx);
    }
  };
  if ((int64_t)blockIdx.x < rows) fetch(blockIdx.x);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        In::unpack(raw[k], v[k]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
      }
    }
    if (row + gridDim.x < rows) fetch(row + gridDim.x);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < EPV; ++e) s += v[k][e];
    const float mu = sum_block_allreduce<THREADS>(s, red[0]) / (float)cols;
    float qs = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (k * THREADS + tid < nvec) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float dlt = v[k][e] - mu;
          qs = fmaf(dlt, dlt, qs);
        }
      }
    }
    const float var = sum_block_allreduce<THREADS>(qs, red[1]) * inv_n;
    if (tid == 0) {
      mean[row] = mu;
      rstd[row] = 1.0f / sqrtf(var + eps);
    }
  }
}

// Layernorm statistics, generic: any cols, any alignment; two passes over
// global memory (sum, then squared deviations about the mean).
template <int THREADS, class In>
__global__ void __launch_bounds__(THREADS)
k_lnstats_gen(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, float eps,
              float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  __shared__ float red[2][THREADS / 32];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const typename In::S *p = x + row * cols;
    float s = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) s += In::load1(p + i);
    const float mu = sum_block_allreduce<THREADS>(s, red[0]) / (float)cols;
    float qs = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) {
      const float dlt = In::load1(p + i) - mu;
      qs = fmaf(dlt, dlt, qs);
    }
    const float var = sum_block_allreduce<THREADS>(qs, red[1]) / (float)cols;
    if (tid == 0) {
      mean[row] = mu;
      rstd[row] = 1.0f / sqrtf(var + eps);
    }
  }
}

// ---------------------------------------------------------------------------
// Layernorm, statistics and rewrite fused ("reduce" page: the rewrite is the
// map pass after the statistics reduce), register-resident row: the
// statistics as in k_lnstats_reg, then y = bf16_rn((x - mean) * rstd *
// gamma + beta) from the registers.  One HBM read of x, one write of y.
// Requires cols % EPV == 0, x / gamma / beta 16-byte aligned, y aligned to
// 2 * EPV bytes.  mean, rstd may be null.
// ---------------------------------------------------------------------------
template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_layernorm_reg(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
                const float *__restrict__ gamma, const float *__restrict__ beta,
                uint16_t *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  constexpr int EPV = In::EPV;
  __shared__ float red[2][THREADS / 32];
  const int tid = threadIdx.x;
  const int nvec = cols / EPV;
  const bool gb32 = aligned32(gamma, beta);
  const float inv_n = 1.0f / (float)cols;
  using W = typename In::W;
  W raw[NV];
  auto fetch = [&](int64_t r) {
    const W *q = reinterpret_cast<const W *>(x + r * (int64_t)cols);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) raw[k] = In::ldv(q + idx);
    }
  };
  if ((int64_t)blockIdx.x < rows) fetch(blockIdx.x);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        In::unpack(raw[k], v[k]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
      }
    }
    if (row + gridDim.x < rows) fetch(row + gridDim.x);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < EPV; ++e) s += v[k][e];
    const float mu = sum_block_allreduce<THREADS>(s, red[0]) / (float)cols;
    float qs = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (k * THREADS + tid < nvec) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float dlt = v[k][e] - mu;
          qs = fmaf(dlt, dlt, qs);
        }
      }
    }
    const float var = sum_block_allreduce<THREADS>(qs, red[1]) * inv_n;
    const float rs = 1.0f / sqrtf(var + eps);
    uint16_t *yr = y + row * (int64_t)cols;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        float g[EPV], b[EPV];
        load_gamma_beta<EPV>(gamma, beta, (int64_t)idx * EPV, gb32, g, b);
        uint32_t pk[EPV / 2];
#pragma unroll
        for (int e = 0; e < EPV; e += 2)
          pk[e / 2] = bf16x2_bits(fmaf((v[k][e] - mu) * rs, g[e], b[e]),
                                  fmaf((v[k][e + 1] - mu) * rs, g[e + 1], b[e + 1]));
        if constexpr (EPV == 8) {
          *reinterpret_cast<uint4 *>(yr + idx * EPV) = make_uint4(pk[0], pk[1 % (EPV / 2)],
                                                                  pk[2 % (EPV / 2)], pk[3 % (EPV / 2)]);
        } else if constexpr (EPV == 4) {
          *reinterpret_cast<uint2 *>(yr + idx * EPV) = make_uint2(pk[0], pk[1 % (EPV / 2)]);
        } else {
          *reinterpret_cast<uint32_t *>(yr + idx * EPV) = pk[0];
        }
      }
    }
    if (tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
  }
}

// Layernorm, generic: any cols, any alignment; statistics in two passes over
// global memory, then the rewrite in a third.
template <int THREADS, class In>
__global__ void __launch_bounds__(THREADS)
k_layernorm_gen(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, float eps,
                const float *__restrict__ gamma, const float *__restrict__ beta,
                uint16_t *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  __shared__ float red[2][THREADS / 32];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const typename In::S *p = x + row * cols;
    float s = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) s += In::load1(p + i);
    const float mu = sum_block_allreduce<THREADS>(s, red[0]) / (float)cols;
    float qs = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) {
      const float dlt = In::load1(p + i) - mu;
      qs = fmaf(dlt, dlt, qs);
    }
    const float rs = 1.0f / sqrtf(sum_block_allreduce<THREADS>(qs, red[1]) / (float)cols + eps);
    uint16_t *yr = y + row * cols;
    for (int64_t i = tid; i < cols; i += THREADS) {
      const __nv_bfloat16 h =
          __float2bfloat16_rn(fmaf((In::load1(p + i) - mu) * rs, __ldg(gamma + i), __ldg(beta + i)));
      yr[i] = *reinterpret_cast<const uint16_t *>(&h);
    }
    if (tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
  }
}

// ---------------------------------------------------------------------------
// Layernorm statistics of rows that do not start 16-byte aligned (a width
// that is not a multiple of the 16-byte vector, or a misaligned x), a CTA
// per row with the row in registers: its head (the elements before its first 16-byte boundary,
// fewer than a vector), its whole 16-byte vectors spread over the threads
// as in the register form, and its tail, one head and one tail element a
// thread.  Each row's head length follows from its own address.
// ---------------------------------------------------------------------------
template <class In>
struct ChunkRow {
  int h, nvec, t;  // head elements, whole vectors, tail elements
  __device__ __forceinline__ ChunkRow(const typename In::S *p, int cols) {
    const int hh = (int)(((16u - ((uint32_t)(uintptr_t)p & 15u)) & 15u) / sizeof(typename In::S));
    h = hh < cols ? hh : cols;
    nvec = (cols - h) / In::EPV;
    t = cols - h - nvec * In::EPV;
  }
};

// The chunked row's raw vectors and its head / tail element of this thread,
// loaded ahead of use (the next row's while the current one is reduced).
template <int THREADS, int NV, class In>
struct ChunkRegs {
  uint4 raw[NV];
  float hv, tv;
  __device__ __forceinline__ ChunkRow<In> fetch(const typename In::S *p, int cols) {
    const ChunkRow<In> g(p, cols);
    const uint4 *q = reinterpret_cast<const uint4 *>(p + g.h);
    const int tid = threadIdx.x;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < g.nvec) raw[k] = ld_stream_u4(q + idx);
    }
    hv = tid < g.h ? In::load1(p + tid) : 0.0f;
    tv = tid < g.t ? In::load1(p + g.h + g.nvec * In::EPV + tid) : 0.0f;
    return g;
  }
};

// The statistics of a chunked row held in v / hv / tv: mean and 1 / sqrt(var
// + eps), two passes over the registers (sum, then squared deviations about
// the mean).
template <int THREADS, int NV, int EPV>
__device__ __forceinline__ void chunk_stats(const float (&v)[NV][EPV], float hv, float tv, int h,
                                            int nvec, int t, int cols, float eps,
                                            float (*red)[THREADS / 32], float &mu, float &rs) {
  const int tid = threadIdx.x;
  float s = hv + tv;
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < EPV; ++e) s += v[k][e];
  mu = sum_block_allreduce<THREADS>(s, red[0]) / (float)cols;
  float qs = 0.0f;
  if (tid < h) qs = (hv - mu) * (hv - mu);
  if (tid < t) qs = fmaf(tv - mu, tv - mu, qs);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (k * THREADS + tid < nvec) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float dlt = v[k][e] - mu;
        qs = fmaf(dlt, dlt, qs);
      }
    }
  }
  rs = 1.0f / sqrtf(sum_block_allreduce<THREADS>(qs, red[1]) / (float)cols + eps);
}

template <int THREADS, int NV, class In>
__device__ __forceinline__ void chunk_unpack(const ChunkRegs<THREADS, NV, In> &cr, int nvec,
                                             float (&v)[NV][In::EPV]) {
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if (k * THREADS + (int)threadIdx.x < nvec) {
      In::unpack(cr.raw[k], v[k]);
    } else {
#pragma unroll
      for (int e = 0; e < In::EPV; ++e) v[k][e] = 0.0f;
    }
  }
}

// Layernorm statistics of chunked rows (any element-aligned x, any cols up
// to THREADS * NV vectors).
template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_lnstats_ck(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
             float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  __shared__ float red[2][THREADS / 32];
  ChunkRegs<THREADS, NV, In> cr;
  ChunkRow<In> g(x, cols);
  if ((int64_t)blockIdx.x < rows) g = cr.fetch(x + (int64_t)blockIdx.x * cols, cols);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    float v[NV][In::EPV];
    chunk_unpack<THREADS, NV, In>(cr, g.nvec, v);
    const float hv = cr.hv, tv = cr.tv;
    const ChunkRow<In> cur = g;
    if (row + gridDim.x < rows) g = cr.fetch(x + (row + gridDim.x) * (int64_t)cols, cols);
    float mu, rs;
    chunk_stats<THREADS, NV, In::EPV>(v, hv, tv, cur.h, cur.nvec, cur.t, cols, eps, red, mu, rs);
    if (threadIdx.x == 0) {
      mean[row] = mu;
      rstd[row] = rs;
    }
  }
}

// Layernorm rewrite of chunked rows: the statistics as k_lnstats_ck (the
// same geometry and fold order, so the same mean / rstd bits), then
// y = (x - mean) * rstd * gamma + beta -> bf16 over the row's head, whole
// vectors and tail.  A vector's columns start at any offset, so gamma and
// beta come from an image each CTA builds once in shared memory: the float2
// (gamma[j], beta[j]) at slot j + j / EPV.  One pad slot per EPV columns
// puts the 16 threads of a half warp, which read columns EPV apart, at
// slots EPV + 1 apart (odd), on 16 distinct 8-byte bank pairs for any head
// offset.  Two elements per packed fp32 instruction; y goes as one vector
// a chunk where it shares x's offset within a 16-byte chunk, element by
// element otherwise.  Dynamic shared memory: ck_image_slots(cols, EPV)
// float2.
__host__ __device__ constexpr int ck_image_slots(int cols, int epv) { return cols + cols / epv + 1; }

template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_layernorm_ck(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
               const float *__restrict__ gamma, const float *__restrict__ beta,
               uint16_t *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  constexpr int EPV = In::EPV;
  extern __shared__ float2 sgb[];
  __shared__ float red[2][THREADS / 32];
  const int tid = threadIdx.x;
  for (int j = tid; j < cols; j += THREADS) sgb[j + j / EPV] = make_float2(__ldg(gamma + j), __ldg(beta + j));
  ChunkRegs<THREADS, NV, In> cr;
  ChunkRow<In> g(x, cols);
  if ((int64_t)blockIdx.x < rows) g = cr.fetch(x + (int64_t)blockIdx.x * cols, cols);
  __syncthreads();
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    float v[NV][EPV];
    chunk_unpack<THREADS, NV, In>(cr, g.nvec, v);
    const float hv = cr.hv, tv = cr.tv;
    const ChunkRow<In> cur = g;
    if (row + gridDim.x < rows) g = cr.fetch(x + (row + gridDim.x) * (int64_t)cols, cols);
    float mu, rs;
    chunk_stats<THREADS, NV, EPV>(v, hv, tv, cur.h, cur.nvec, cur.t, cols, eps, red, mu, rs);
    if (tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
    uint16_t *yr = y + row * (int64_t)cols;
    auto put = [&](int j, float xv) {
      const float2 gb = sgb[j + j / EPV];
      const __nv_bfloat16 ob = __float2bfloat16_rn(fmaf((xv - mu) * rs, gb.x, gb.y));
      yr[j] = *reinterpret_cast<const uint16_t *>(&ob);
    };
    if (tid < cur.h) put(tid, hv);
    if (tid < cur.t) put(cur.h + cur.nvec * EPV + tid, tv);
    const bool vst = ((uintptr_t)(yr + cur.h) & (2 * EPV - 1)) == 0;
    const uint64_t mu2 = f2_pack(mu, mu), rs2 = f2_pack(rs, rs);
    // every whole vector starts at column h (mod EPV): its element e sits at
    // slot e + dq[e] past the vector's first column's slot
    int dq[EPV];
#pragma unroll
    for (int e = 0; e < EPV; ++e) dq[e] = e + (e >= EPV - cur.h ? 1 : 0);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx >= cur.nvec) continue;
      const int j0 = cur.h + idx * EPV;
      const float2 *q = sgb + j0 + j0 / EPV;
      uint32_t pk[EPV / 2];
#pragma unroll
      for (int i = 0; i < EPV / 2; ++i) {
        const float2 g0 = q[dq[2 * i]], g1 = q[dq[2 * i + 1]];
        float lo, hi;
        f2_unpack(f2_fma(f2_mul(f2_sub(f2_pack(v[k][2 * i], v[k][2 * i + 1]), mu2), rs2),
                         f2_pack(g0.x, g1.x), f2_pack(g0.y, g1.y)),
                  lo, hi);
        pk[i] = bf16x2_bits(lo, hi);
      }
      uint16_t *p = yr + j0;
      if (vst) {
        if constexpr (EPV == 8) *reinterpret_cast<uint4 *>(p) = make_uint4(pk[0], pk[1 % (EPV / 2)], pk[2 % (EPV / 2)], pk[3 % (EPV / 2)]);
        else *reinterpret_cast<uint2 *>(p) = make_uint2(pk[0], pk[1 % (EPV / 2)]);
      } else {
#pragma unroll
        for (int i = 0; i < EPV / 2; ++i) {
          p[2 * i] = (uint16_t)(pk[i] & 0xffffu);
          p[2 * i + 1] = (uint16_t)(pk[i] >> 16);
        }
      }
    }
  }
}

// Softmax of chunked rows (rows that are not 16-byte aligned, up to 1024
// vectors): the row held as head + whole 16-byte vectors + tail as in
// k_lnstats_ck, the next row's loaded while the current one is reduced;
// each thread's (max, sum) over its elements, one block combine of the
// pairs, then y = e^(x - M) / S in fp32: one 32-byte (bf16 input) or
// 16-byte store a vector where y's offset allows, element by element
// otherwise.  Empty slots hold -inf, so their terms are exactly 0.
template <int THREADS, int NV, class In>
__global__ void __launch_bounds__(THREADS)
k_softmax_ck(const typename In::S *__restrict__ x, int64_t rows, int cols, float *__restrict__ y) {
  pdl_begin();
  constexpr int EPV = In::EPV;
  __shared__ float red_m[THREADS / 32 + 1], red_s[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  ChunkRegs<THREADS, NV, In> cr;
  ChunkRow<In> g(x, cols);
  if ((int64_t)blockIdx.x < rows) g = cr.fetch(x + (int64_t)blockIdx.x * cols, cols);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const ChunkRow<In> cur = g;
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (k * THREADS + tid < cur.nvec) {
        In::unpack(cr.raw[k], v[k]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = -INFINITY;
      }
    }
    float hv = tid < cur.h ? cr.hv : -INFINITY, tv = tid < cur.t ? cr.tv : -INFINITY;
    if (row + gridDim.x < rows) g = cr.fetch(x + (row + gridDim.x) * (int64_t)cols, cols);
    float m = fmaxf(hv, tv);
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < EPV; ++e) m = fmaxf(m, v[k][e]);
    float s = 0.0f;
    if (m != -INFINITY) {
      const float mb = m * kLog2e;
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float p = ex2_approx(fmaf(v[k][e], kLog2e, -mb));
          v[k][e] = p;
          s += p;
        }
      hv = ex2_approx(fmaf(hv, kLog2e, -mb));
      tv = ex2_approx(fmaf(tv, kLog2e, -mb));
      s += hv + tv;
    } else {
      // every element this thread holds is -inf: e^(x - M) = 0
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
      hv = tv = 0.0f;
    }
    float M = m, S = s;
    ms_block_allreduce<THREADS>(M, S, red_m, red_s);
    const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S);
    float *yr = y + row * (int64_t)cols;
    if (tid < cur.h) yr[tid] = hv * f;
    if (tid < cur.t) yr[cur.h + cur.nvec * EPV + tid] = tv * f;
    const uintptr_t ya = (uintptr_t)(yr + cur.h);
    const int vw = ya % (4 * EPV) == 0 ? 2 : (ya % 16 == 0 ? 1 : 0);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx >= cur.nvec) continue;
      float *p = yr + cur.h + (int64_t)idx * EPV;
      float o[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) o[e] = v[k][e] * f;
      if constexpr (EPV == 8) {
        if (vw == 2) {
          st_stream_v8(p, o);
          continue;
        }
      }
      if (vw) {
#pragma unroll
        for (int e = 0; e < EPV; e += 4) st_stream_v4(p + e, o[e], o[e + 1], o[e + 2], o[e + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) p[e] = o[e];
      }
    }
    __syncthreads();
  }
}

template <class K>
int persistent_grid(K kernel, int threads, int64_t rows, const DevInfo &d, size_t smem = 0) {
  const int nb = occupancy_blocks((const void *)kernel, threads, smem, d.device);
  const int64_t cap = (int64_t)nb * d.sm_count;
  return (int)(rows < cap ? rows : cap);
}

// Registers per thread hold NV vectors; NV is the smallest power of two
// with THREADS * NV * EPV >= cols, up to 8.
inline int pick_nv(int64_t nvec) {
  for (int nv = 1; nv <= 8; nv <<= 1)
    if ((int64_t)kRowThreads * nv >= nvec) return nv;
  return 0;
}
// Geometry of the chunked kernels (k_lnstats_ck, k_layernorm_ck) for rows
// of nvec vectors: CTAs of kChunkThreads threads holding NV = 1, 2 or 4
// vectors each up to 4 * kChunkThreads vectors, then kRowThreads x 4 (the
// return value 8), up to 1024; 0 beyond.  128 threads rather than 256: a
// row's two block reductions cost each thread about as much as its two
// vectors of arithmetic, so fewer threads with more vectors each issue
// fewer instructions a row, and one more CTA fits an SM (16384 x 4099
// bf16 statistics / rewrite 0.57 / 0.60 -> 0.70 / 0.64, 65536 x 1029 fp32
// 0.40 / 0.39 -> 0.59 / 0.53; rows of 513 to 1024 vectors unchanged).
constexpr int kChunkThreads = 128;
inline int chunk_geometry(int64_t nvec) {
  for (int nv = 1; nv <= 4; nv <<= 1)
    if ((int64_t)kChunkThreads * nv >= nvec) return nv;
  return nvec <= (int64_t)kRowThreads * 4 ? 8 : 0;
}
// Layernorm rows of more than 4 vectors per thread (1025 to 2048 vectors)
// run with kRowWideThreads threads and 4 vectors each instead of 256 x 8:
// the rewrite measured 11-20% faster (at 8 vectors a thread, with gamma and
// beta, too few warps stayed resident).  The statistics take the same
// geometry, 3-14% slower on their own, so that both fold in the same order
// and return the same mean and rstd bits.
constexpr int kRowWideThreads = 512;
// Rows of 1025 to 1536 vectors take 288 or 384 threads (4 vectors each)
// instead of 512, so that a row just past 1024 vectors does not leave half
// the slots empty (16384 x 4100 bf16: 1025 8-byte vectors).
inline int wide_threads(int64_t nvec) { return nvec <= 1152 ? 288 : (nvec <= 1536 ? 384 : 512); }

// ---------------------------------------------------------------------------
// Split-K tier of the two-pass row operations ("reduce" page, split-K tier;
// "cluster_allreduce" page, two-slot mode).  A cluster of C CTAs per row;
// CTA r owns slice r of the row (a multiple of 8 elements, shifted like the
// reduce tier's so that every slice but the first starts 16-byte aligned).
// The first pass reads the slice from HBM; a second read of the same bytes
// is served by L2 (this tier only runs for a few long rows).  Each row takes
// two cluster combines, back to back on two slots with no tail sync between
// them and one terminal cluster sync:
//   softmax:   one pass of per-thread online (max, sum) over the slice, the
//              CTA pair; combine the maxima -> M; rescale the CTA sum to M;
//              combine the sums -> S; then y = e^(x - M) / S over the slice.
//   layernorm: CTA sum -> combine -> mean; CTA sum of (x - mean)^2 ->
//              combine -> var; rstd (and the rewrite).
// Every CTA folds the partials in rank order, so every CTA holds the same
// M, S (mean, var) bits.  The passes read 8-element vectors where the slice
// is 16-byte aligned, element by element otherwise.
// ---------------------------------------------------------------------------
// Folds the 8-element vectors v = tid, tid + THREADS, ... < nv of ps, in that
// order: st = f(st, v, e).  U vectors per thread are loaded back to back
// before the first is used (raw words first, unpacked after), so U * 16 bytes
// (bf16) or U * 32 bytes (fp32) per thread are in flight; the order of the
// calls, and so every fold done in f, is the same as a one-at-a-time loop.
// The state is passed by value so that it stays in registers.
#ifndef RR_ROWSK_UNROLL
#define RR_ROWSK_UNROLL 4
#endif
#ifndef RR_ROWSK_THREADS
#define RR_ROWSK_THREADS 512
#endif
template <class In, int NW>
__device__ __forceinline__ void unpack8(const uint4 (&w)[NW], float (&o)[8]) {
  if constexpr (NW == 1) {
    In::unpack(w[0], o);
  } else {
    o[0] = __uint_as_float(w[0].x); o[1] = __uint_as_float(w[0].y);
    o[2] = __uint_as_float(w[0].z); o[3] = __uint_as_float(w[0].w);
    o[4] = __uint_as_float(w[1].x); o[5] = __uint_as_float(w[1].y);
    o[6] = __uint_as_float(w[1].z); o[7] = __uint_as_float(w[1].w);
  }
}
template <int THREADS, int U, class In, class St, class F>
__device__ __forceinline__ St fold_vectors(const typename In::S *ps, int64_t nv, St st, F f) {
  constexpr int NW = In::EPV == 8 ? 1 : 2;  // 16-byte words per vector
  int64_t v = threadIdx.x;
  for (; v + (int64_t)(U - 1) * THREADS < nv; v += (int64_t)U * THREADS) {
    uint4 w[U][NW];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NW; ++k)
        w[u][k] = ld_stream_u4(ps + (v + (int64_t)u * THREADS) * 8 + 4 * k);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float e[8];
      unpack8<In, NW>(w[u], e);
      st = f(st, v + (int64_t)u * THREADS, e);
    }
  }
  for (; v < nv; v += THREADS) {
    uint4 w[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = ld_stream_u4(ps + v * 8 + 4 * k);
    float e[8];
    unpack8<In, NW>(w, e);
    st = f(st, v, e);
  }
  return st;
}

// MODE: kModeSoftmax (y fp32), kModeStats (mean, rstd), kModeLayernorm
// (mean, rstd and the rewrite ybf = bf16((x - mean) * rstd * gamma + beta)).
template <int THREADS, class In, int MODE>
__global__ void __launch_bounds__(THREADS)
k_rowwise_splitk(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, float eps,
                 float *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 uint16_t *__restrict__ ybf) {
  pdl_begin();
  using S = typename In::S;
  __shared__ float red_m[THREADS / 32 + 1], red_s[THREADS / 32 + 1];
  __shared__ float slot[2][2];
  const int tid = threadIdx.x;
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t row = cluster_id_x();
  const S *p = x + row * cols;
  const int64_t chunk = ((cols + C - 1) / C + 7) & ~int64_t(7);
  const int64_t mis = (int64_t)((16u - ((uint32_t)(uintptr_t)p & 15u)) & 15u) / (int64_t)sizeof(S);
  auto bound = [&](int64_t k) -> int64_t {
    if (k == 0) return 0;
    if (k >= (int64_t)C) return cols;
    const int64_t b = k * chunk + mis - (mis ? 8 : 0);
    return b < 0 ? 0 : (b > cols ? cols : b);
  };
  const int64_t b0 = bound(r), b1 = bound(r + 1);
  const int64_t n = b1 > b0 ? b1 - b0 : 0;
  const S *ps = p + b0;
  const int64_t nv = ((uintptr_t)ps % 16 == 0) ? (n >> 3) : 0;  // vectors; then a scalar tail

  if (MODE == kModeSoftmax) {
    const float2 ms = fold_vectors<THREADS, RR_ROWSK_UNROLL, In>(
        ps, nv, make_float2(-INFINITY, 0.0f), [](float2 st, int64_t, const float (&e)[8]) {
          float cm = e[0];
#pragma unroll
          for (int j = 1; j < 8; ++j) cm = fmaxf(cm, e[j]);
          if (cm > st.x) {
            st.y = (st.x == -INFINITY) ? 0.0f : st.y * ex2_approx((st.x - cm) * kLog2e);
            st.x = cm;
          }
          if (st.x != -INFINITY) {
            const float mb = st.x * kLog2e;
#pragma unroll
            for (int j = 0; j < 8; ++j) st.y += ex2_approx(fmaf(e[j], kLog2e, -mb));
          }
          return st;
        });
    float m = ms.x, s = ms.y;
    for (int64_t i = nv * 8 + tid; i < n; i += THREADS) ms_combine(m, s, In::load1(ps + i), 1.0f);
    ms_block_allreduce<THREADS>(m, s, red_m, red_s);  // the CTA pair, in every thread
    float v1[1] = {m}, M[1];
    cluster_allreduce<MaxF32, 1>(slot[0], v1, C, /*tail_sync=*/false, M);  // combine 1
    float v2[1] = {(m == -INFINITY) ? 0.0f : s * ex2_approx((m - M[0]) * kLog2e)}, Ssum[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, Ssum);  // combine 2
    const float inv = 1.0f / Ssum[0];
    const float mb = M[0] * kLog2e;
    float *yr = y + row * cols + b0;
    const bool vy = ((uintptr_t)yr % 16 == 0);
    const float Mx = M[0];
    fold_vectors<THREADS, RR_ROWSK_UNROLL, In>(
        ps, nv, 0, [=](int st, int64_t v, const float (&x8)[8]) {
          float e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            e[j] = (Mx == -INFINITY) ? 0.0f : ex2_approx(fmaf(x8[j], kLog2e, -mb)) * inv;
          if (vy) {
            st_stream_v4(yr + v * 8, e[0], e[1], e[2], e[3]);
            st_stream_v4(yr + v * 8 + 4, e[4], e[5], e[6], e[7]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) yr[v * 8 + j] = e[j];
          }
          return st;
        });
    for (int64_t i = nv * 8 + tid; i < n; i += THREADS)
      yr[i] = (M[0] == -INFINITY) ? 0.0f : ex2_approx(fmaf(In::load1(ps + i), kLog2e, -mb)) * inv;
  } else {
    float acc = fold_vectors<THREADS, RR_ROWSK_UNROLL, In>(
        ps, nv, 0.0f, [](float a, int64_t, const float (&e)[8]) {
#pragma unroll
          for (int j = 0; j < 8; ++j) a += e[j];
          return a;
        });
    for (int64_t i = nv * 8 + tid; i < n; i += THREADS) acc += In::load1(ps + i);
    acc = block_reduce<SumF32, THREADS>(acc, red_s);
    float v1[1] = {acc}, tot[1];
    cluster_allreduce<SumF32, 1>(slot[0], v1, C, /*tail_sync=*/false, tot);  // combine 1
    const float mu = tot[0] / (float)cols;
    float q = fold_vectors<THREADS, RR_ROWSK_UNROLL, In>(
        ps, nv, 0.0f, [=](float a, int64_t, const float (&e)[8]) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float d = e[j] - mu;
            a = fmaf(d, d, a);
          }
          return a;
        });
    for (int64_t i = nv * 8 + tid; i < n; i += THREADS) {
      const float d = In::load1(ps + i) - mu;
      q = fmaf(d, d, q);
    }
    __syncthreads();  // red_s is reused
    q = block_reduce<SumF32, THREADS>(q, red_s);
    float v2[1] = {q}, tq[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, tq);  // combine 2
    const float rs = 1.0f / sqrtf(tq[0] / (float)cols + eps);
    if (r == 0 && tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
    if (MODE == kModeLayernorm) {
      uint16_t *yr = ybf + row * cols + b0;
      const bool vy = ((uintptr_t)yr % 16 == 0) && ((uintptr_t)(gamma + b0) % 16 == 0) &&
                      ((uintptr_t)(beta + b0) % 16 == 0);
      fold_vectors<THREADS, RR_ROWSK_UNROLL, In>(
          ps, nv, 0, [=](int st, int64_t v, const float (&e)[8]) {
        if (vy) {
          const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + b0 + v * 8));
          const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + b0 + v * 8 + 4));
          const float4 c0 = __ldg(reinterpret_cast<const float4 *>(beta + b0 + v * 8));
          const float4 c1 = __ldg(reinterpret_cast<const float4 *>(beta + b0 + v * 8 + 4));
          uint4 o;
          o.x = bf16x2_bits(fmaf((e[0] - mu) * rs, g0.x, c0.x), fmaf((e[1] - mu) * rs, g0.y, c0.y));
          o.y = bf16x2_bits(fmaf((e[2] - mu) * rs, g0.z, c0.z), fmaf((e[3] - mu) * rs, g0.w, c0.w));
          o.z = bf16x2_bits(fmaf((e[4] - mu) * rs, g1.x, c1.x), fmaf((e[5] - mu) * rs, g1.y, c1.y));
          o.w = bf16x2_bits(fmaf((e[6] - mu) * rs, g1.z, c1.z), fmaf((e[7] - mu) * rs, g1.w, c1.w));
          *reinterpret_cast<uint4 *>(yr + v * 8) = o;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int64_t i = v * 8 + j;
            const __nv_bfloat16 h = __float2bfloat16_rn(
                fmaf((e[j] - mu) * rs, __ldg(gamma + b0 + i), __ldg(beta + b0 + i)));
            yr[i] = *reinterpret_cast<const uint16_t *>(&h);
          }
        }
        return st;
      });
      for (int64_t i = nv * 8 + tid; i < n; i += THREADS) {
        const __nv_bfloat16 h = __float2bfloat16_rn(
            fmaf((In::load1(ps + i) - mu) * rs, __ldg(gamma + b0 + i), __ldg(beta + b0 + i)));
        yr[i] = *reinterpret_cast<const uint16_t *>(&h);
      }
    }
  }
  // the second combine dropped its tail sync: retire both slots before exit
  cluster_sync();
}

template <class In, int MODE>
int launch_rowwise_splitk(const void *xv, int64_t rows, int64_t cols, float eps, float *y,
                          float *mean, float *rstd, const float *gamma, const float *beta,
                          uint16_t *ybf, int C, cudaStream_t s, const DevInfo &d) {
  using S = typename In::S;
  constexpr int T = RR_ROWSK_THREADS;
  auto kern = k_rowwise_splitk<T, In, MODE>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (C > 1 && occupancy_clusters((const void *)kern, T, 0, C, d.device) < 1)
    return RR_ERR_UNSUPPORTED;
  if (rows * C > 0x7fffffffLL) return RR_ERR_INVALID;
  if (log_enabled())
    std::fprintf(stderr, "rr: %s split-K rows=%lld cols=%lld C=%d\n",
                 MODE == kModeSoftmax ? "softmax" : (MODE == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, C);
  return cuda_status(launch_kernel(kern, dim3((unsigned)(rows * C)), dim3(T), 0, s, C,
                                   (const S *)xv, rows, cols, eps, y, mean, rstd, gamma, beta,
                                   ybf));
}

// Tier of a two-pass row op on a device (its SM count, and its largest
// cluster: RR_MAX_CLUSTER caps it, no cluster launch makes it 1).
template <class In>
inline RowPlan rowwise_pick(int64_t rows, int64_t cols, bool vec, int tier, int C,
                            const DevInfo &d, int mode, const void *x, const void *out,
                            bool half = false, bool grid_ok = false) {
  const int cap = cluster_cap() < 16 ? cluster_cap() : 16;
  const int dt = In::EPV == 8 ? RR_BF16 : RR_F32;
  return plan_rowwise(rows, cols, dt, vec, mode, tier, C, d.sm_count, d.cluster_launch ? cap : 1,
                      rowwise_warp_out_vec(mode, dt, x, out), half && tier == RR_TIER_AUTO,
                      grid_ok && tier == RR_TIER_AUTO);
}

// rr_last_tier's code: tier | (width & 0xff) << 8 | flags << 16 |
// (width >> 8) << 19, flags 1 staged, 2 ring, 4 grid.
inline int tier_code(int tier, int width, int flags) {
  return tier | ((width & 0xff) << 8) | (flags << 16) | (((width >> 8) & 0xff) << 19);
}
constexpr int kFlagStaged = 1, kFlagRing = 2, kFlagGrid = 4;
constexpr int kChunkBit = 1 << 27;  // the chunked register form (k_*_ck)
constexpr int kTwoPassBit = 1 << 28;  // the rewrite's two-pass form

// The grid form's plan for a call: forced (w.splits), automatic with the
// caller's workspace (falling back to the plan without one when it is too
// small), or none.  grid_ok: the operands meet the form's alignment.
template <class In>
inline RowPlan rowwise_pick_ws(int64_t rows, int64_t cols, bool vec, int tier, int C,
                               const DevInfo &d, int mode, const void *x, const void *out,
                               bool half, bool grid_ok, const RowWs &w) {
  grid_ok = grid_ok && w.ws != nullptr && (uintptr_t)w.ws % 16 == 0;
  if (w.splits > 0) {
    if (!grid_ok) return RowPlan{-1, 0, false};
    RowPlan p{RR_TIER_SPLITK, w.splits, false};
    p.grid = true;
    return p;
  }
  RowPlan p = rowwise_pick<In>(rows, cols, vec, tier, C, d, mode, x, out, half, grid_ok);
  if ((p.grid && rowgrid_ws_bytes(rows, p.width) > w.bytes) ||
      (p.twopass && rowtwopass_ws_bytes(rows) > w.bytes))
    p = rowwise_pick<In>(rows, cols, vec, tier, C, d, mode, x, out, half, false);
  return p;
}

// The 8-byte vector element type of an input type.
template <class In> struct HalfOf;
template <> struct HalfOf<InBF16> { using T = InBF16h; };
template <> struct HalfOf<InF32> { using T = InF32h; };

template <class In>
int softmax_impl(const void *xv, int64_t rows, int64_t cols, float *y, cudaStream_t s,
                 const DevInfo &d, int *tier_out, int tier, int C, const RowWs &w) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const uintptr_t ax = (uintptr_t)xv, ay = (uintptr_t)y;
  const int64_t nvec = cols / In::EPV;
  const bool vec = (cols % In::EPV == 0) && ax % 16 == 0 &&
                   (In::EPV == 8 ? ay % 32 == 0 : ay % 16 == 0);
  using H = typename HalfOf<In>::T;
  const bool half = cols % H::EPV == 0 && ax % 8 == 0 && ay % (H::EPV * 4) == 0;
  const RowPlan pk = rowwise_pick_ws<In>(rows, cols, vec, tier, C, d, kModeSoftmax, xv, y, half,
                                         vec && cols % 8 == 0 && ay % 32 == 0, w);
  if (pk.tier < 0) return RR_ERR_UNSUPPORTED;
  *tier_out = tier_code(pk.tier, pk.width, pk.staged ? kFlagStaged : 0);
  if (pk.grid) {
    *tier_out = tier_code(pk.tier, pk.width, kFlagGrid);
    return launch_rowgrid(kModeSoftmax, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, 0.0f, y,
                          nullptr, nullptr, nullptr, nullptr, nullptr, pk.width, w.ws, w.bytes, s,
                          d);
  }
  if (pk.ring && ay % 32 == 0) {
    int Cl = pk.width;
    const int st = launch_rowwise_ring(kModeSoftmax, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows,
                                       cols, 0.0f, y, nullptr, nullptr, nullptr, nullptr, nullptr,
                                       pk.width, tier == RR_TIER_AUTO, &Cl, s, d);
    *tier_out = tier_code(pk.tier, Cl, kFlagRing);
    return st;
  }
  if (pk.staged)
    return launch_rowwise_staged(kModeSoftmax, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols,
                                 0.0f, y, nullptr, nullptr, nullptr, nullptr, nullptr, pk.width, vec, s, d);
  if (pk.tier == RR_TIER_SPLITK)
    return launch_rowwise_splitk<In, kModeSoftmax>(xv, rows, cols, 0.0f, y, nullptr, nullptr,
                                                   nullptr, nullptr, nullptr, pk.width, s, d);
  if (pk.tier == RR_TIER_WARP)
    return (vec ? launch_rowwise_warp : launch_rowwise_warp_mis)(kModeSoftmax, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols,
                               0.0f, y, nullptr, nullptr, nullptr, nullptr, nullptr, pk.width, s, d);
  if (pk.chunk) {
    *tier_out |= kChunkBit;
#define RR_SM_CK(T, NV)                                                        \
  {                                                                            \
    auto k = k_softmax_ck<T, NV, In>;                                          \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, y); \
  }
    switch (chunk_geometry(cols / In::EPV)) {
      case 1: RR_SM_CK(kChunkThreads, 1) break;
      case 2: RR_SM_CK(kChunkThreads, 2) break;
      case 4: RR_SM_CK(kChunkThreads, 4) break;
      case 8: RR_SM_CK(kRowThreads, 4) break;
      default: return RR_ERR_UNSUPPORTED;
    }
#undef RR_SM_CK
    return cuda_status(cudaGetLastError());
  }
  const bool reg = vec && pick_nv(nvec) > 0;
  if (pk.half) {
#define RR_SM_REGH(T, NV)                                                      \
  {                                                                            \
    auto k = k_softmax_reg<T, NV, H>;                                          \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, y); \
  }
    switch (pick_nv(cols / H::EPV)) {
      case 1: RR_SM_REGH(kRowThreads, 1) break;
      case 2: RR_SM_REGH(kRowThreads, 2) break;
      case 4: RR_SM_REGH(kRowThreads, 4) break;
      default: RR_SM_REGH(kRowThreads, 8) break;
    }
#undef RR_SM_REGH
  } else if (reg) {
#define RR_SM_REG(T, NV)                                                       \
  {                                                                            \
    auto k = k_softmax_reg<T, NV, In>;                                         \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, y); \
  }
    switch (pick_nv(nvec)) {
      case 1: RR_SM_REG(kRowThreads, 1) break;
      case 2: RR_SM_REG(kRowThreads, 2) break;
      case 4: RR_SM_REG(kRowThreads, 4) break;
      default: RR_SM_REG(kRowThreads, 8) break;  // (rows this long are staged)
    }
#undef RR_SM_REG
  } else {
    auto k = k_softmax_gen<kRowThreads, In>;
    launch_kernel(k, dim3(persistent_grid(k, kRowThreads, rows, d)), dim3(kRowThreads), 0, s, 0, x, rows, cols, y);
  }
  return cuda_status(cudaGetLastError());
}

template <class In>
int lnstats_impl(const void *xv, int64_t rows, int64_t cols, float eps, float *mean,
                 float *rstd, cudaStream_t s, const DevInfo &d, int *tier_out, int tier, int C,
                 const RowWs &w) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const int64_t nvec = cols / In::EPV;
  const bool vec = (cols % In::EPV == 0) && ((uintptr_t)xv % 16 == 0);
  using H = typename HalfOf<In>::T;
  const bool half = cols % H::EPV == 0 && (uintptr_t)xv % 8 == 0;
  const RowPlan pk = rowwise_pick_ws<In>(rows, cols, vec, tier, C, d, kModeStats, xv, nullptr,
                                         half, vec && cols % 8 == 0, w);
  if (pk.tier < 0) return RR_ERR_UNSUPPORTED;
  *tier_out = tier_code(pk.tier, pk.width, pk.staged ? kFlagStaged : 0);
  if (pk.grid) {
    *tier_out = tier_code(pk.tier, pk.width, kFlagGrid);
    return launch_rowgrid(kModeStats, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, eps,
                          nullptr, mean, rstd, nullptr, nullptr, nullptr, pk.width, w.ws, w.bytes,
                          s, d);
  }
  if (pk.ring) {
    int Cl = pk.width;
    const int st = launch_rowwise_ring(kModeStats, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols,
                                       eps, nullptr, mean, rstd, nullptr, nullptr, nullptr,
                                       pk.width, tier == RR_TIER_AUTO, &Cl, s, d);
    *tier_out = tier_code(pk.tier, Cl, kFlagRing);
    return st;
  }
  if (pk.staged)
    return launch_rowwise_staged(kModeStats, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, eps,
                                 nullptr, mean, rstd, nullptr, nullptr, nullptr, pk.width, vec, s, d);
  if (pk.tier == RR_TIER_SPLITK)
    return launch_rowwise_splitk<In, kModeStats>(xv, rows, cols, eps, nullptr, mean, rstd,
                                                 nullptr, nullptr, nullptr, pk.width, s, d);
  if (pk.tier == RR_TIER_WARP)
    return (vec ? launch_rowwise_warp : launch_rowwise_warp_mis)(kModeStats, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, eps,
                               nullptr, mean, rstd, nullptr, nullptr, nullptr, pk.width, s, d);
  if (pk.chunk) {
    *tier_out |= kChunkBit;
#define RR_LN_CK(T, NV)                                                        \
  {                                                                            \
    auto k = k_lnstats_ck<T, NV, In>;                                          \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, eps, mean, rstd); \
  }
    switch (chunk_geometry(cols / In::EPV)) {  // the rewrite's geometry: the same bits
      case 1: RR_LN_CK(kChunkThreads, 1) break;
      case 2: RR_LN_CK(kChunkThreads, 2) break;
      case 4: RR_LN_CK(kChunkThreads, 4) break;
      case 8: RR_LN_CK(kRowThreads, 4) break;
      default: return RR_ERR_UNSUPPORTED;
    }
#undef RR_LN_CK
    return cuda_status(cudaGetLastError());
  }
  const bool reg = vec && pick_nv(nvec) > 0;
  if (pk.half) {
#define RR_LN_REGH(T, NV)                                                      \
  {                                                                            \
    auto k = k_lnstats_reg<T, NV, H>;                                          \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, eps, mean, rstd); \
  }
    switch (pick_nv(cols / H::EPV)) {  // the rewrite's geometry: the same bits
      case 1: RR_LN_REGH(kRowThreads, 1) break;
      case 2: RR_LN_REGH(kRowThreads, 2) break;
      case 4: RR_LN_REGH(kRowThreads, 4) break;
      default:
        if (wide_threads(cols / H::EPV) == 288) RR_LN_REGH(288, 4)
        else if (wide_threads(cols / H::EPV) == 384) RR_LN_REGH(384, 4)
        else RR_LN_REGH(kRowWideThreads, 4)
        break;
    }
#undef RR_LN_REGH
  } else if (reg) {
#define RR_LN_REG(T, NV)                                                       \
  {                                                                            \
    auto k = k_lnstats_reg<T, NV, In>;                                         \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0, x, rows, (int)cols, eps, mean, rstd); \
  }
    switch (pick_nv(nvec)) {  // the rewrite's geometry: the same fold order, the same bits
      case 1: RR_LN_REG(kRowThreads, 1) break;
      case 2: RR_LN_REG(kRowThreads, 2) break;
      case 4: RR_LN_REG(kRowThreads, 4) break;
      default:
        if (wide_threads(nvec) == 288) RR_LN_REG(288, 4)
        else if (wide_threads(nvec) == 384) RR_LN_REG(384, 4)
        else RR_LN_REG(kRowWideThreads, 4)
        break;
    }
#undef RR_LN_REG
  } else {
    auto k = k_lnstats_gen<kRowThreads, In>;
    launch_kernel(k, dim3(persistent_grid(k, kRowThreads, rows, d)), dim3(kRowThreads), 0, s, 0, x, rows, cols, eps, mean, rstd);
  }
  return cuda_status(cudaGetLastError());
}

template <class In>
int layernorm_impl(const void *xv, int64_t rows, int64_t cols, float eps, const float *gamma,
                   const float *beta, uint16_t *y, float *mean, float *rstd, cudaStream_t s,
                   const DevInfo &d, int *tier_out, int tier, int C, const RowWs &w) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const int64_t nvec = cols / In::EPV;
  const bool vec = (cols % In::EPV == 0) && ((uintptr_t)xv % 16 == 0) &&
                   ((uintptr_t)gamma % 16 == 0) && ((uintptr_t)beta % 16 == 0) &&
                   ((uintptr_t)y % (2 * In::EPV) == 0);
  using H = typename HalfOf<In>::T;
  const bool half = cols % H::EPV == 0 && (uintptr_t)xv % 8 == 0 &&
                    (uintptr_t)gamma % (H::EPV * 4) == 0 && (uintptr_t)beta % (H::EPV * 4) == 0 &&
                    (uintptr_t)y % (H::EPV * 2) == 0;
  const RowPlan pk = rowwise_pick_ws<In>(rows, cols, vec, tier, C, d, kModeLayernorm, xv, y, half,
                                         vec && cols % 8 == 0 && (uintptr_t)y % 16 == 0, w);
  if (pk.tier < 0) return RR_ERR_UNSUPPORTED;
  *tier_out = tier_code(pk.tier, pk.width, pk.staged ? kFlagStaged : 0);
  if (pk.grid) {
    *tier_out = tier_code(pk.tier, pk.width, kFlagGrid);
    return launch_rowgrid(kModeLayernorm, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, eps,
                          nullptr, mean, rstd, gamma, beta, y, pk.width, w.ws, w.bytes, s, d);
  }
  if (pk.twopass) {
    // the statistics into mean / rstd where asked for, else the workspace
    float *mu = mean ? mean : (float *)w.ws;
    float *rs = rstd ? rstd : (float *)w.ws + rows;
    int Cl = 1;
    int st = launch_rowwise_ring(kModeStats, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, eps,
                                 nullptr, mu, rs, nullptr, nullptr, nullptr, 1, true, &Cl, s, d);
    if (st != RR_OK) return st;
    *tier_out = tier_code(RR_TIER_BLOCK, 1, 0) | kTwoPassBit;
    return launch_ln_apply(In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols, mu, rs, gamma, beta, y,
                           s, d);
  }
  if (pk.ring && (uintptr_t)y % 16 == 0) {
    int Cl = pk.width;
    const int st = launch_rowwise_ring(kModeLayernorm, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows,
                                       cols, eps, nullptr, mean, rstd, gamma, beta, y, pk.width,
                                       tier == RR_TIER_AUTO, &Cl, s, d);
    *tier_out = tier_code(pk.tier, Cl, kFlagRing);
    return st;
  }
  if (pk.staged)
    return launch_rowwise_staged(kModeLayernorm, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols,
                                 eps, nullptr, mean, rstd, gamma, beta, y, pk.width, vec, s, d);
  if (pk.tier == RR_TIER_SPLITK)
    return launch_rowwise_splitk<In, kModeLayernorm>(xv, rows, cols, eps, nullptr, mean, rstd,
                                                     gamma, beta, y, pk.width, s, d);
  if (pk.tier == RR_TIER_WARP)
    return (vec ? launch_rowwise_warp : launch_rowwise_warp_mis)(kModeLayernorm, In::EPV == 8 ? RR_BF16 : RR_F32, xv, rows, cols,
                               eps, nullptr, mean, rstd, gamma, beta, y, pk.width, s, d);
  if (pk.chunk) {
    *tier_out |= kChunkBit;
    const size_t smem = (size_t)ck_image_slots((int)cols, In::EPV) * sizeof(float2);
#define RR_LNF_CK(T, NV)                                                       \
  {                                                                            \
    auto k = k_layernorm_ck<T, NV, In>;                                        \
    const cudaError_t e =                                                      \
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (e != cudaSuccess) return cuda_status(e);                               \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d, smem)), dim3(T), smem, s, 0, \
        x, rows, (int)cols, eps, gamma, beta, y, mean, rstd);                  \
  }
    switch (chunk_geometry(cols / In::EPV)) {  // the statistics' geometry: the same bits
      case 1: RR_LNF_CK(kChunkThreads, 1) break;
      case 2: RR_LNF_CK(kChunkThreads, 2) break;
      case 4: RR_LNF_CK(kChunkThreads, 4) break;
      case 8: RR_LNF_CK(kRowThreads, 4) break;
      default: return RR_ERR_UNSUPPORTED;
    }
#undef RR_LNF_CK
    return cuda_status(cudaGetLastError());
  }
  const bool reg = vec && pick_nv(nvec) > 0;
  if (pk.half) {
#define RR_LNF_REGH(T, NV)                                                     \
  {                                                                            \
    auto k = k_layernorm_reg<T, NV, H>;                                        \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0,   \
        x, rows, (int)cols, eps, gamma, beta, y, mean, rstd);                  \
  }
    switch (pick_nv(cols / H::EPV)) {
      case 1: RR_LNF_REGH(kRowThreads, 1) break;
      case 2: RR_LNF_REGH(kRowThreads, 2) break;
      case 4: RR_LNF_REGH(kRowThreads, 4) break;
      default:
        if (wide_threads(cols / H::EPV) == 288) RR_LNF_REGH(288, 4)
        else if (wide_threads(cols / H::EPV) == 384) RR_LNF_REGH(384, 4)
        else RR_LNF_REGH(kRowWideThreads, 4)
        break;
    }
#undef RR_LNF_REGH
  } else if (reg) {
#define RR_LNF_REG(T, NV)                                                      \
  {                                                                            \
    auto k = k_layernorm_reg<T, NV, In>;                                       \
    launch_kernel(k, dim3(persistent_grid(k, T, rows, d)), dim3(T), 0, s, 0,   \
        x, rows, (int)cols, eps, gamma, beta, y, mean, rstd);                  \
  }
    switch (pick_nv(nvec)) {
      case 1: RR_LNF_REG(kRowThreads, 1) break;
      case 2: RR_LNF_REG(kRowThreads, 2) break;
      case 4: RR_LNF_REG(kRowThreads, 4) break;
      default:
        if (wide_threads(nvec) == 288) RR_LNF_REG(288, 4)
        else if (wide_threads(nvec) == 384) RR_LNF_REG(384, 4)
        else RR_LNF_REG(kRowWideThreads, 4)
        break;
    }
#undef RR_LNF_REG
  } else {
    auto k = k_layernorm_gen<kRowThreads, In>;
    launch_kernel(k, dim3(persistent_grid(k, kRowThreads, rows, d)), dim3(kRowThreads), 0, s, 0, x, rows, cols, eps, gamma,
                                                                        beta, y, mean, rstd);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

// Split-K cluster size for a two-pass row op: the smallest power of two >= 2
// that puts a CTA on every SM, at most max_cluster (<= 16); 0 when the tier
// does not apply (a few long rows only).
static int rowwise_splitk_cluster(int64_t rows, int64_t cols, int sm_count, int max_cluster) {
  if (max_cluster < 2 || rows < 1 || rows >= sm_count || cols < 16384) return 0;
  int c = 2;
  while (2 * c <= max_cluster && (int64_t)c * rows < sm_count) c *= 2;
  return c;
}

// Staged rows: the automatic choice stages softmax rows of more than 1024
// 16-byte vectors and the layernorm's beyond the register form (2048; the
// register form measured better there for them, worse for softmax, whose
// 8-vector register rows at 256 threads hold 64 floats and its exponentials
// per thread); forced split-K stages its slices when RR_ROW_STAGED_SPLITK
// and they fit.
constexpr int64_t kRowStagedMinVec[3] = {1024, kRowRegMaxVec, kRowRegMaxVec};
constexpr int64_t kRowThreadsHost = 256;  // kRowThreads, for the host plan
// Shortest rows the automatic plan gives the grid form (a few rows only).
constexpr int64_t kRowGridMinCols = 16384;
// Rows that are not 16-byte aligned and not held in the chunked register
// form (below) are staged beyond these lengths in 16-byte vectors (softmax,
// statistics, rewrite), shorter ones take the scalar form.  Measured
// against that form and the split-K fallback: staging wins for softmax
// from the shortest rows tried (4100 bf16: 5026 against 4315 GB/s; 8193:
// 6396 against 1620), for the statistics from about 1024 vectors, for the
// rewrite from about 2048.
constexpr int64_t kRowStagedMinVecMis[3] = {32, 1024, 2048};
#ifndef RR_ROW_STAGED_SPLITK
#define RR_ROW_STAGED_SPLITK 0
#endif

RowPlan plan_rowwise(int64_t rows, int64_t cols, int in_dtype, bool vec, int mode, int tier,
                     int C, int sm_count, int max_cluster, bool out_vec, bool half, bool grid_ok) {
  const bool rewrite = mode == kModeLayernorm;
  const int64_t elt = in_dtype == RR_BF16 ? 2 : 4;
  const int64_t nvec = vec ? cols * elt / 16 : 0;
  const int64_t row_vecs = cols * elt / 16;  // the row's length in 16-byte vectors
  // staged slices of C CTAs fit shared memory (misaligned rows stage up to
  // 8 elements more)
  auto stage_fits = [&](int c) {
    return (rowwise_staged_chunk(cols, c) + (vec ? 0 : 8)) * elt <= kStageMaxBytes;
  };
  const int warp_min_rows_per_sm = rewrite ? kRowWarpMinRowsPerSMRewrite : kRowWarpMinRowsPerSM;
  // the streamed ring form (rowring.cu): aligned rows of whole 8-element
  // units; softmax and the rewrite read each slice twice, the second time
  // from L2, so only while the rows in flight fit there
  const bool ring_ok = vec && cols % 8 == 0;
  auto ring_fits = [&](int64_t inflight_rows) {
    return mode == kModeStats || inflight_rows * cols * elt <= kRingL2Bytes;
  };
  // a few long rows: the ring for softmax and the statistics; the rewrite
  // keeps the global-memory split-K form, whose 16-CTA clusters spread the
  // per-row gamma / beta reads (8 bytes an element, from L2) over more SMs
  // (16 x 1M bf16: 35 against 48 us)
  const bool ring_few = mode != kModeLayernorm;
  const int64_t staged_min = vec ? kRowStagedMinVec[mode] : kRowStagedMinVecMis[mode];
  // the statistics and the rewrite of rows that are not 16-byte aligned:
  // the chunked register form (head + 16-byte vectors + tail) up to 1024
  // vectors, where they would otherwise take the scalar two-pass form (the
  // statistics: 16384 x 4099 bf16 0.41 -> 0.70, 16384 x 4095 fp32 0.58 ->
  // 1.00; beyond 1024 vectors staging measured ahead, 4096 x 16383 bf16 0.68
  // against 0.43; the rewrite, gamma / beta from a padded image in shared
  // memory: 16384 x 4099 bf16 0.44 -> 0.64, 16384 x 8196 0.47 -> 0.64,
  // 16384 x 4095 fp32 0.61 -> 0.79, 65536 x 1029 fp32 0.32 -> 0.53)
  // softmax too, up to 4096 elements (512 bf16 / 1024 fp32 vectors), when
  // its output shares x's offset within a 16-byte chunk (vector stores),
  // rather than staging (16384 x 4099 bf16 0.74 -> 0.90, 16384 x 2057 0.47
  // -> 0.64, 65536 x 1029 fp32 0.40 -> 0.73; 8192 x 8191 bf16 staged 0.94
  // against 0.80, an x base off the output's offset 0.38 against 0.27)
  const bool chunk_ok =
      !vec && (mode != kModeSoftmax ? row_vecs <= kRowStagedMinVecMis[kModeStats]
                                    : out_vec && row_vecs <= (in_dtype == RR_BF16 ? 512 : 1024));
  if (tier == RR_TIER_BLOCK) {
    const bool st = row_vecs > staged_min && stage_fits(1);
    if (!st && chunk_ok) {
      RowPlan p{RR_TIER_BLOCK, 1, false};
      p.chunk = true;
      return p;
    }
    return {RR_TIER_BLOCK, 1, st};
  }
  if (tier == RR_TIER_WARP) {
    const int L = vec ? rowwise_warp_lanes(nvec, C, rewrite)
                      : rowwise_warp_mis_lanes(cols, in_dtype, mode, out_vec, C);
    return L ? RowPlan{RR_TIER_WARP, L, false} : RowPlan{-1, 0, false};
  }
  if (tier == RR_TIER_SPLITK) {
    if (C == 0) C = rowwise_splitk_cluster(rows, cols, sm_count, max_cluster);
    if (C == 0) C = 2;
    if (C > 1 && C > max_cluster) return {-1, 0, false};
    const int64_t inflight = 2 * (int64_t)sm_count / C;
    if (ring_ok && ring_fits(rows < inflight ? rows : inflight))
      return {RR_TIER_SPLITK, C, false, true};
    const bool st = RR_ROW_STAGED_SPLITK && stage_fits(C);
    return {RR_TIER_SPLITK, C, st};
  }
  // a few long rows, with a workspace: the grid form (rowgrid.cu), the
  // slices on every SM and no clusters
  if (grid_ok && ring_ok && rows >= 1 && rows < sm_count && cols >= kRowGridMinCols) {
    RowPlan p{RR_TIER_SPLITK, rowgrid_splits(rows, cols, sm_count), false};
    p.grid = true;
    return p;
  }
  const int c = rowwise_splitk_cluster(rows, cols, sm_count, max_cluster);
  if (c > 0) {
    // a few long rows: with the ring, a cluster of as many CTAs as there
    // are SMs per row (any size up to 16), one CTA per SM
    if (ring_few && ring_ok && ring_fits(rows)) {
      int cr = (int)(sm_count / rows);
      if (cr > 16) cr = 16;
      if (cr > max_cluster) cr = max_cluster;
      if (cr <= 1) return {RR_TIER_BLOCK, 1, false, true};  // a CTA per row
      return {RR_TIER_SPLITK, cr, false, true};
    }
    const bool st = RR_ROW_STAGED_SPLITK && stage_fits(c);
    return {RR_TIER_SPLITK, c, st};
  }
  if (rows >= (int64_t)warp_min_rows_per_sm * sm_count) {
    const int L = vec ? rowwise_warp_lanes(nvec, 0, rewrite)
                      : rowwise_warp_mis_lanes(cols, in_dtype, mode, out_vec, 0);
    if (L) return {RR_TIER_WARP, L, false};
  }
  // the statistics of rows of 128 KiB and more: a CTA per row, streamed once
  // through the ring (measured against staging a CTA per row: 608 x 262144
  // bf16 0.88 against 0.49 of the copy bandwidth, 4096 x 32768 0.80 against
  // 0.87 -- shorter rows stage)
  if (mode == kModeStats && ring_ok && row_vecs > kRowRegMaxVec && cols * elt >= (128 << 10))
    return {RR_TIER_BLOCK, 1, false, true};
  // rows whose base is only 8-byte aligned (widths of 4k bf16 / 2k fp32
  // elements that are not 8k / 4k): the register form read as 8-byte
  // vectors, up to 2048 of them, rather than staging or the scalar form
  // (softmax up to 1024 of them: beyond, staging measured ahead, 16384 x 4100
  // bf16 0.74 against 0.57)
  if (!vec && half &&
      cols / (in_dtype == RR_BF16 ? 4 : 2) <= (int64_t)kRowThreadsHost * (mode == kModeSoftmax ? 4 : 8))
    return RowPlan{RR_TIER_BLOCK, 1, false, false, true};
  if (chunk_ok) {
    RowPlan p{RR_TIER_BLOCK, 1, false};
    p.chunk = true;
    return p;
  }
  // the rewrite of many long rows, with a workspace: the statistics through
  // the ring (a CTA per row), then a rewrite pass that reads x again with
  // gamma / beta held over a group of rows (rowgrid.cu), rather than staging
  // the rows, whose rewrite reloads gamma / beta (8 bytes an element) for
  // every row
  if (rewrite && grid_ok && ring_ok && rows >= sm_count && cols * elt >= kRowTwoPassMinBytes) {
    RowPlan p{RR_TIER_BLOCK, 1, false};
    p.twopass = true;
    return p;
  }
  if (row_vecs > staged_min) {
    const int sc = rowwise_staged_cluster(cols, in_dtype, max_cluster, vec);
    if (sc == 1) return {RR_TIER_BLOCK, 1, true};
    // the statistics only read the row: past clusters of 4 the split-K pass
    // over global memory (its second read served by L2) came out ahead
    if (sc > 1 && !(mode == kModeStats && sc > 4)) return {RR_TIER_SPLITK, sc, true};
  }
  // long rows that cannot be staged (not vector-aligned, or more than 16
  // slices): split-K over global memory, slices of at most 128 KiB, rather
  // than the block tier's scalar two-pass form
  const int64_t row_bytes = cols * elt;
  if (row_bytes > 16 * kRowStagedMinVec[mode] && max_cluster >= 2) {
    int c2 = 2;
    while (c2 < max_cluster && c2 < 16 && row_bytes / c2 > 128 * 1024) c2 *= 2;
    return {RR_TIER_SPLITK, c2, false};
  }
  return {RR_TIER_BLOCK, 1, false};
}

int launch_layernorm(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                     const float *gamma, const float *beta, uint16_t *y, float *mean, float *rstd,
                     cudaStream_t s, const DevInfo &d, int *tier_out, int tier, int C,
                     const RowWs &w) {
  if (in_dtype == RR_BF16)
    return layernorm_impl<InBF16>(x, rows, cols, eps, gamma, beta, y, mean, rstd, s, d, tier_out,
                                  tier, C, w);
  return layernorm_impl<InF32>(x, rows, cols, eps, gamma, beta, y, mean, rstd, s, d, tier_out,
                               tier, C, w);
}

int launch_softmax(const void *x, int64_t rows, int64_t cols, int in_dtype, float *out,
                   cudaStream_t s, const DevInfo &d, int *tier_out, int tier, int C,
                   const RowWs &w) {
  if (in_dtype == RR_BF16)
    return softmax_impl<InBF16>(x, rows, cols, out, s, d, tier_out, tier, C, w);
  return softmax_impl<InF32>(x, rows, cols, out, s, d, tier_out, tier, C, w);
}

int launch_layernorm_stats(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                           float *mean, float *rstd, cudaStream_t s, const DevInfo &d,
                           int *tier_out, int tier, int C, const RowWs &w) {
  if (in_dtype == RR_BF16)
    return lnstats_impl<InBF16>(x, rows, cols, eps, mean, rstd, s, d, tier_out, tier, C, w);
  return lnstats_impl<InF32>(x, rows, cols, eps, mean, rstd, s, d, tier_out, tier, C, w);
}

}  // namespace rr
