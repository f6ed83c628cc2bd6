// rowwise.cu -- the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise): softmax (pass 1 reduces the online-softmax
// (max, sum) monoid, pass 2 is a stateless map that writes exp(x - m) / s)
// and the layernorm statistics (mean, then the variance about the mean, both
// block reduces over the on-chip row).
//
// Fast path: one CTA per row with the whole row held in registers, so the
// row is read from HBM exactly once.  Generic path (any width, any
// alignment): the row is streamed from global memory once per pass.
#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

#ifndef RR_ROW_THREADS
#define RR_ROW_THREADS 256
#endif
constexpr int kRowThreads = RR_ROW_THREADS;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Input element types: bf16 (held as its raw 16 bits) or fp32.
struct InBF16 {
  using S = unsigned short;
  static constexpr int EPV = 8;  // elements per 16-byte vector
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&o)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(u[i] << 16);
      o[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ float load1(const S *p) {
    return __uint_as_float(((uint32_t)__ldg(p)) << 16);
  }
};
struct InF32 {
  using S = float;
  static constexpr int EPV = 4;
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&o)[4]) {
    o[0] = __uint_as_float(w.x); o[1] = __uint_as_float(w.y);
    o[2] = __uint_as_float(w.z); o[3] = __uint_as_float(w.w);
  }
  static __device__ __forceinline__ float load1(const S *p) { return __ldg(p); }
};

// ---------------------------------------------------------------------------
// The online-softmax (max, sum) monoid: (m1, s1) + (m2, s2) =
// (M, s1 * e^(m1 - M) + s2 * e^(m2 - M)), M = max(m1, m2), identity
// (-inf, 0).  A side whose max is -inf contributes 0 (no -inf - -inf NaN).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  const float a = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - M) * kLog2e);
  const float b = (m2 == -INFINITY) ? 0.0f : s2 * ex2_approx((m2 - M) * kLog2e);
  m = M;
  s = a + b;
}

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

// Block sum; every thread receives the result.
template <int THREADS>
__device__ __forceinline__ float sum_block_allreduce(float v, float *red) {
  constexpr int NW = THREADS / 32;
  v = block_reduce<SumF32, THREADS>(v, red);
  if (threadIdx.x == 0) red[NW] = v;
  __syncthreads();
  v = red[NW];
  __syncthreads();
  return v;
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
  constexpr int EPV = In::EPV;
  __shared__ float red_m[THREADS / 32 + 1], red_s[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  const int nvec = cols / EPV;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint4 *q = reinterpret_cast<const uint4 *>(x + row * (int64_t)cols);
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        In::unpack(ld_stream_u4(q + idx), v[k]);
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
    }
    float M = m, S = s;
    ms_block_allreduce<THREADS>(M, S, red_m, red_s);
    const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S);
    float *yr = y + row * (int64_t)cols;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) {
        if (EPV == 8) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = v[k][e % EPV] * f;
          st_stream_v8(yr + (int64_t)idx * EPV, o);
        } else {
          st_stream_v4(yr + (int64_t)idx * EPV, v[k][0] * f, v[k][1 % EPV] * f,
                       v[k][2 % EPV] * f, v[k][3 % EPV] * f);
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
  constexpr int EPV = In::EPV;
  __shared__ float red[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  const int nvec = cols / EPV;
  const float inv_n = 1.0f / (float)cols;
  uint4 raw[NV];
  auto fetch = [&](int64_t r) {
    const uint4 *q = reinterpret_cast<const uint4 *>(x + r * (int64_t)cols);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * THREADS + tid;
      if (idx < nvec) raw[k] = ld_stream_u4(q + idx);
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
    const float mu = sum_block_allreduce<THREADS>(s, red) / (float)cols;
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
    const float var = sum_block_allreduce<THREADS>(qs, red) * inv_n;
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
  __shared__ float red[THREADS / 32 + 1];
  const int tid = threadIdx.x;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const typename In::S *p = x + row * cols;
    float s = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) s += In::load1(p + i);
    const float mu = sum_block_allreduce<THREADS>(s, red) / (float)cols;
    float qs = 0.0f;
    for (int64_t i = tid; i < cols; i += THREADS) {
      const float dlt = In::load1(p + i) - mu;
      qs = fmaf(dlt, dlt, qs);
    }
    const float var = sum_block_allreduce<THREADS>(qs, red) / (float)cols;
    if (tid == 0) {
      mean[row] = mu;
      rstd[row] = 1.0f / sqrtf(var + eps);
    }
  }
}

template <class K>
int persistent_grid(K kernel, int threads, int64_t rows, const DevInfo &d) {
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess || nb < 1)
    nb = 1;
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

template <class In>
int softmax_impl(const void *xv, int64_t rows, int64_t cols, float *y, cudaStream_t s,
                 const DevInfo &d, int *tier_out) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const uintptr_t ax = (uintptr_t)xv, ay = (uintptr_t)y;
  const int64_t nvec = cols / In::EPV;
  const bool reg = (cols % In::EPV == 0) && ax % 16 == 0 &&
                   (In::EPV == 8 ? ay % 32 == 0 : ay % 16 == 0) && pick_nv(nvec) > 0;
  if (reg) {
    *tier_out = RR_TIER_BLOCK;
#define RR_SM_REG(NV)                                                          \
  {                                                                            \
    auto k = k_softmax_reg<kRowThreads, NV, In>;                               \
    k<<<persistent_grid(k, kRowThreads, rows, d), kRowThreads, 0, s>>>(x, rows, (int)cols, y); \
  }
    switch (pick_nv(nvec)) {
      case 1: RR_SM_REG(1) break;
      case 2: RR_SM_REG(2) break;
      case 4: RR_SM_REG(4) break;
      default: RR_SM_REG(8) break;
    }
#undef RR_SM_REG
  } else {
    *tier_out = RR_TIER_BLOCK;
    auto k = k_softmax_gen<kRowThreads, In>;
    k<<<persistent_grid(k, kRowThreads, rows, d), kRowThreads, 0, s>>>(x, rows, cols, y);
  }
  return cuda_status(cudaGetLastError());
}

template <class In>
int lnstats_impl(const void *xv, int64_t rows, int64_t cols, float eps, float *mean,
                 float *rstd, cudaStream_t s, const DevInfo &d, int *tier_out) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const int64_t nvec = cols / In::EPV;
  const bool reg = (cols % In::EPV == 0) && ((uintptr_t)xv % 16 == 0) && pick_nv(nvec) > 0;
  *tier_out = RR_TIER_BLOCK;
  if (reg) {
#define RR_LN_REG(NV)                                                          \
  {                                                                            \
    auto k = k_lnstats_reg<kRowThreads, NV, In>;                               \
    k<<<persistent_grid(k, kRowThreads, rows, d), kRowThreads, 0, s>>>(x, rows, (int)cols, eps, mean, rstd); \
  }
    switch (pick_nv(nvec)) {
      case 1: RR_LN_REG(1) break;
      case 2: RR_LN_REG(2) break;
      case 4: RR_LN_REG(4) break;
      default: RR_LN_REG(8) break;
    }
#undef RR_LN_REG
  } else {
    auto k = k_lnstats_gen<kRowThreads, In>;
    k<<<persistent_grid(k, kRowThreads, rows, d), kRowThreads, 0, s>>>(x, rows, cols, eps, mean, rstd);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

int launch_softmax(const void *x, int64_t rows, int64_t cols, int in_dtype, float *out,
                   cudaStream_t s, const DevInfo &d, int *tier_out) {
  if (in_dtype == RR_BF16) return softmax_impl<InBF16>(x, rows, cols, out, s, d, tier_out);
  return softmax_impl<InF32>(x, rows, cols, out, s, d, tier_out);
}

int launch_layernorm_stats(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                           float *mean, float *rstd, cudaStream_t s, const DevInfo &d,
                           int *tier_out) {
  if (in_dtype == RR_BF16)
    return lnstats_impl<InBF16>(x, rows, cols, eps, mean, rstd, s, d, tier_out);
  return lnstats_impl<InF32>(x, rows, cols, eps, mean, rstd, s, d, tier_out);
}

}  // namespace rr
