// rowgrid.cu -- the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise: softmax, layernorm statistics, layernorm rewrite)
// for a few long rows, spread over every SM without clusters.
//
// The split-K tier cuts a row into slices folded by the CTAs of a cluster
// and combined through distributed shared memory; with fewer rows than SMs
// those clusters cover only part of the GPU (a cluster must sit inside one
// GPC).  Here the slices go to G CTAs of a plain grid, CTA (row, g) taking
// slice g, and their partial states pass through a caller-owned workspace
// to a second launch in stream order, as the page's multi-cluster split-K
// passes cluster partials:
//
//   k_rowgrid_part         CTA (row, g) folds slice g of the row into one
//                          monoid state -- the online-softmax (max, sum)
//                          pair, or the layernorm's (count, mean, M2) --
//                          and stores it in ws[row * G + g];
//   k_rowgrid_softmax_out  CTA (row, g) folds the row's G states and writes
//                          slice g of the output, reading the slice again;
//   k_rowgrid_ln_out       CTA (column block, row group; 512 threads) folds
//                          the states of its rows and rewrites its columns of
//                          them, gamma and beta read once per row group;
//   k_rowgrid_stats_fin    a warp per row folds its states into mean, rstd.
//
// (One-launch forms -- the statistics folded by each row's last CTA in, and
// softmax / the rewrite as a cooperative launch whose CTAs wait for their
// row's states, with the slice re-read from L2 or staged in shared memory
// by bulk copies -- measured slower on every shape tried: 16 x 1M bf16
// softmax 22.5 against 21.0 us, statistics 12.2 against 10.4 us.)
//
// Every fold of a row's G states takes one order -- lane l merges states
// l, l + 32, ... in turn, then the lanes merge by an xor butterfly with the
// lower lane on the left -- so every CTA of a row, the statistics kernel and
// every run get the same bits.  Within a slice, a thread folds rounds of
// 8-element units (units tid, tid + 256, ...; 96 bytes a thread a round):
// softmax as the online update (the round's maximum, then its terms against
// the running maximum); layernorm two-pass about the round's own mean,
// merged into the thread's state with the update of Chan, Golub and
// LeVeque, so variances are taken about means at every level and the row
// is read once.  The warps' states are merged in warp order.  (Measured on
// 16 x 1M bf16: a copy of the statistics' first launch with its arithmetic
// replaced by an XOR of the loaded words took 9.8 against 10.5 us, so the
// arithmetic is not what bounds it; a shifted single pass (sums of x - K
// and (x - K)^2, K the thread's first element) took 10.2 us but subtracts
// squared sums, and an L2 bulk prefetch of each slice at the kernel's start
// 10.8 us.  Neither was kept.)
#include <climits>
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"
#include "rowwise.cuh"

namespace rr {
namespace {

constexpr int kGridThreads = 256;
constexpr int kGridWarps = kGridThreads / 32;
constexpr int kGridCtasPerSm = 4;    // CTAs per SM the slices aim at
// Units (8 elements) a thread has in flight: 96 bytes of x either way.
template <class In>
__host__ __device__ constexpr int grid_unroll() {
  return In::EPV == 8 ? 6 : 3;
}

// 8 elements of a 16-byte aligned slice: one 16-byte word of bf16, two of
// fp32, read past L1.
template <class In>
struct GridUnit {
  static constexpr int NW = In::EPV == 8 ? 1 : 2;
  uint4 w[NW];
  // unit u of the 16-byte words q, with L2 eviction policy pol
  __device__ __forceinline__ void load(const uint4 *q, int u, uint64_t pol) {
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = ld_stream_u4_hint(q + (size_t)u * NW + k, pol);
  }
  // elements 2k, 2k + 1 as packed fp32 pair k
  __device__ __forceinline__ void pairs(uint64_t (&e2)[4]) const {
    if constexpr (NW == 1) {
      e2[0] = bf16x2_to_f2(w[0].x);
      e2[1] = bf16x2_to_f2(w[0].y);
      e2[2] = bf16x2_to_f2(w[0].z);
      e2[3] = bf16x2_to_f2(w[0].w);
    } else {
      e2[0] = ((uint64_t)w[0].y << 32) | w[0].x;
      e2[1] = ((uint64_t)w[0].w << 32) | w[0].z;
      e2[2] = ((uint64_t)w[1].y << 32) | w[1].x;
      e2[3] = ((uint64_t)w[1].w << 32) | w[1].z;
    }
  }
};

// One round of nv units (a prefix of un) into the thread's (max, sum): the
// round's maximum first, the running sum rescaled once if it rises, then
// the round's terms e^(x - m) against the running maximum.
template <class In, int U = grid_unroll<In>()>
__device__ __forceinline__ void round_ms(const GridUnit<In> (&un)[U], int nv, float &m, float &s) {
  float cm = -INFINITY;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    if (k < nv) {
      uint64_t e2[4];
      un[k].pairs(e2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float lo, hi;
        f2_unpack(e2[q], lo, hi);
        cm = fmaxf(cm, fmaxf(lo, hi));
      }
    }
  }
  if (cm > m) {
    s = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - cm) * kLog2e);
    m = cm;
  }
  if (m == -INFINITY) return;
  const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
  const uint64_t nmb2 = f2_pack(-m * kLog2e, -m * kLog2e);
  uint64_t aa = 0, ab = 0;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    if (k < nv) {
      uint64_t e2[4];
      un[k].pairs(e2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float lo, hi;
        f2_unpack(f2_fma(e2[q], l2e2, nmb2), lo, hi);
        const uint64_t t = f2_pack(ex2_approx(lo), ex2_approx(hi));
        if (q & 1) ab = f2_add(ab, t); else aa = f2_add(aa, t);
      }
    }
  }
  float alo, ahi;
  f2_unpack(f2_add(aa, ab), alo, ahi);
  s += alo + ahi;
}

// One round of nv units as a (count, mean, M2) leaf, two-pass about its own
// mean, two elements per instruction.
template <class In, int U = grid_unroll<In>()>
__device__ __forceinline__ Chan round_chan(const GridUnit<In> (&un)[U], int nv) {
  uint64_t sa = 0, sb = 0;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    if (k < nv) {
      uint64_t e2[4];
      un[k].pairs(e2);
      sa = f2_add(sa, e2[0]);
      sb = f2_add(sb, e2[1]);
      sa = f2_add(sa, e2[2]);
      sb = f2_add(sb, e2[3]);
    }
  }
  float slo, shi;
  f2_unpack(f2_add(sa, sb), slo, shi);
  const float lm = __fdividef(slo + shi, (float)(8 * nv));
  const uint64_t nlm = f2_pack(-lm, -lm);
  uint64_t qa = 0, qb = 0;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    if (k < nv) {
      uint64_t e2[4];
      un[k].pairs(e2);
      uint64_t d = f2_add(e2[0], nlm);
      qa = f2_fma(d, d, qa);
      d = f2_add(e2[1], nlm);
      qb = f2_fma(d, d, qb);
      d = f2_add(e2[2], nlm);
      qa = f2_fma(d, d, qa);
      d = f2_add(e2[3], nlm);
      qb = f2_fma(d, d, qb);
    }
  }
  float qlo, qhi;
  f2_unpack(f2_add(qa, qb), qlo, qhi);
  return Chan{(uint32_t)(8 * nv), lm, qlo + qhi};
}

// Slice g of a row: [g * chunk, min((g + 1) * chunk, cols)), chunk a
// multiple of 8 (empty past the row's end).
struct Slice {
  int64_t b0, nu;  // first element, whole 8-element units
};
__device__ __forceinline__ Slice grid_slice(int64_t cols, int64_t chunk, int g) {
  int64_t b0 = (int64_t)g * chunk;
  if (b0 > cols) b0 = cols;
  const int64_t b1 = b0 + chunk < cols ? b0 + chunk : cols;
  return Slice{b0, (b1 - b0) >> 3};
}

// A warp folds the G states of `row` in the fixed order described at the
// top of the file; every lane returns the same bits.
__device__ __forceinline__ void fold_row_ms(const uint4 *__restrict__ ws, int64_t row, int G,
                                            float &m, float &s) {
  const int lane = threadIdx.x & 31;
  m = -INFINITY;
  s = 0.0f;
  for (int g = lane; g < G; g += 32) {
    const uint4 w = __ldcg(ws + row * G + g);
    ms_combine(m, s, __uint_as_float(w.x), __uint_as_float(w.y));
  }
  ms_warp<32>(m, s);
}
__device__ __forceinline__ Chan fold_row_chan(const uint4 *__restrict__ ws, int64_t row, int G) {
  const int lane = threadIdx.x & 31;
  Chan c{0u, 0.0f, 0.0f};
  for (int g = lane; g < G; g += 32) {
    const uint4 w = __ldcg(ws + row * G + g);
    c = chan_merge(c, Chan{w.x, __uint_as_float(w.y), __uint_as_float(w.z)});
  }
  return chan_warp<32>(c);
}

__device__ __forceinline__ float rstd_of(const Chan &c, int64_t cols, float eps) {
  return 1.0f / sqrtf(c.m2 / (float)cols + eps);
}

// The threads' states merged into the CTA's: each warp by the xor
// butterfly, then the warps in warp order by thread 0, which gets the
// result.
template <int MODE>
__device__ __forceinline__ uint4 finish_state(float m, float sm, Chan st,
                                              uint4 (&wst)[kGridWarps]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if constexpr (MODE == kModeSoftmax) {
    ms_warp<32>(m, sm);
    if (lane == 0) wst[warp] = make_uint4(__float_as_uint(m), __float_as_uint(sm), 0u, 0u);
  } else {
    st = chan_warp<32>(st);
    if (lane == 0) wst[warp] = make_uint4(st.n, __float_as_uint(st.mean), __float_as_uint(st.m2), 0u);
  }
  __syncthreads();
  uint4 w = wst[0];
  if (tid == 0) {
    if constexpr (MODE == kModeSoftmax) {
      float a = __uint_as_float(w.x), b = __uint_as_float(w.y);
      for (int k = 1; k < kGridWarps; ++k)
        ms_combine(a, b, __uint_as_float(wst[k].x), __uint_as_float(wst[k].y));
      w = make_uint4(__float_as_uint(a), __float_as_uint(b), 0u, 0u);
    } else {
      Chan t{w.x, __uint_as_float(w.y), __uint_as_float(w.z)};
      for (int k = 1; k < kGridWarps; ++k)
        t = chan_merge(t, Chan{wst[k].x, __uint_as_float(wst[k].y), __uint_as_float(wst[k].z)});
      w = make_uint4(t.n, __float_as_uint(t.mean), __float_as_uint(t.m2), 0u);
    }
  }
  return w;
}

// Phase 1 of CTA (row, g): slice g folded into the CTA's state, returned
// to thread 0 (MODE kModeSoftmax: the (max, sum) pair, otherwise (count,
// mean, M2)).  q: the slice's 16-byte words, nu its units; pol the L2
// policy of the loads.
template <class In, int MODE>
__device__ __forceinline__ uint4 fold_slice(const uint4 *q, int nu, uint64_t pol,
                                            uint4 (&wst)[kGridWarps]) {
  const int tid = threadIdx.x;
  float m = -INFINITY, sm = 0.0f;
  Chan st{0u, 0.0f, 0.0f};
  constexpr int U = grid_unroll<In>();
  int u0 = tid;
  // whole rounds, no predicates
  for (; u0 + (U - 1) * kGridThreads < nu; u0 += kGridThreads * U) {
    GridUnit<In> un[U];
#pragma unroll
    for (int k = 0; k < U; ++k) un[k].load(q, u0 + k * kGridThreads, pol);
    if constexpr (MODE == kModeSoftmax) round_ms<In>(un, U, m, sm);
    else st = chan_merge(st, round_chan<In>(un, U));
  }
  // the last, partial round
  if (u0 < nu) {
    GridUnit<In> un[U];
    int nv = 0;
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (u0 + k * kGridThreads < nu) {
        un[k].load(q, u0 + k * kGridThreads, pol);
        nv = k + 1;
      }
    }
    if constexpr (MODE == kModeSoftmax) round_ms<In>(un, nv, m, sm);
    else st = chan_merge(st, round_chan<In>(un, nv));
  }
  return finish_state<MODE>(m, sm, st, wst);
}

// First launch: the CTA's state into ws[row * G + g].  Grid rows * G, x
// 16-byte aligned, cols a multiple of 8.  KEEP: x is read again, keep its
// lines in L2 ahead of other traffic.
template <class In, int MODE, bool KEEP>
__global__ void __launch_bounds__(kGridThreads, kGridCtasPerSm)
k_rowgrid_part(const typename In::S *__restrict__ x, int64_t cols, int G, int64_t chunk,
               uint4 *__restrict__ ws) {
  pdl_begin();
  __shared__ uint4 wst[kGridWarps];
  const int64_t row = blockIdx.x / G;
  const int g = (int)(blockIdx.x - row * G);
  const Slice sl = grid_slice(cols, chunk, g);
  const uint4 *q = reinterpret_cast<const uint4 *>(x + row * cols + sl.b0);
  const uint4 w = fold_slice<In, MODE>(q, (int)sl.nu,
                                       KEEP ? l2_evict_last_policy() : l2_evict_first_policy(), wst);
  pdl_release();
  if (threadIdx.x == 0) ws[blockIdx.x] = w;
}

// Softmax output of slice g of the row: y = e^(x - M) / S, fp32, y 32-byte
// aligned.  An all -inf row (M = -inf) gives zeros.
template <class In>
__global__ void __launch_bounds__(kGridThreads, kGridCtasPerSm)
k_rowgrid_softmax_out(const typename In::S *__restrict__ x, int64_t cols, int G, int64_t chunk,
                      const uint4 *__restrict__ ws, float *__restrict__ y) {
  pdl_begin();
  __shared__ float res[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x / G;
  const int g = (int)(blockIdx.x - row * G);
  const Slice sl = grid_slice(cols, chunk, g);
  const uint4 *q = reinterpret_cast<const uint4 *>(x + row * cols + sl.b0);
  const int nu = (int)sl.nu;
  constexpr int U = grid_unroll<In>();
  const uint64_t pol = l2_evict_first_policy();  // x's last read
  // the first round's loads go out before the wait for the row's result
  GridUnit<In> un0[U];
#pragma unroll
  for (int k = 0; k < U; ++k)
    if (tid + k * kGridThreads < nu) un0[k].load(q, tid + k * kGridThreads, pol);
  if (warp == 0) {
    float m, s;
    fold_row_ms(ws, row, G, m, s);
    if (lane == 0) {
      res[0] = m;
      res[1] = 1.0f / s;
    }
  }
  __syncthreads();
  const float Mx = res[0], inv = res[1];
  const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
  const uint64_t nmb2 = f2_pack(-Mx * kLog2e, -Mx * kLog2e), inv2 = f2_pack(inv, inv);
  float *yp = y + row * cols + sl.b0;
  const bool dead = Mx == -INFINITY;
  auto emit = [&](const GridUnit<In> &un, int u) {
    uint64_t e2[4];
    float o[8];
    un.pairs(e2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float lo, hi;
      f2_unpack(f2_fma(e2[k], l2e2, nmb2), lo, hi);
      f2_unpack(f2_mul(f2_pack(ex2_approx(lo), ex2_approx(hi)), inv2), o[2 * k], o[2 * k + 1]);
    }
    if (dead) {
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = 0.0f;
    }
    st_stream_v8(yp + (size_t)u * 8, o);
  };
#pragma unroll
  for (int k = 0; k < U; ++k)
    if (tid + k * kGridThreads < nu) emit(un0[k], tid + k * kGridThreads);
  int u0 = tid + kGridThreads * U;
  for (; u0 + (U - 1) * kGridThreads < nu; u0 += kGridThreads * U) {
    GridUnit<In> un[U];
#pragma unroll
    for (int k = 0; k < U; ++k) un[k].load(q, u0 + k * kGridThreads, pol);
#pragma unroll
    for (int k = 0; k < U; ++k) emit(un[k], u0 + k * kGridThreads);
  }
  if (u0 < nu) {
    GridUnit<In> un[U];
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (u0 + k * kGridThreads < nu) un[k].load(q, u0 + k * kGridThreads, pol);
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (u0 + k * kGridThreads < nu) emit(un[k], u0 + k * kGridThreads);
  }
}

// Layernorm rewrite: CTA (bx, by) of kLnThreads threads takes units
// bx * kLnThreads + tid of rows [by * RB, min((by + 1) * RB, rows)); ybf,
// gamma, beta 16-byte aligned.  Dynamic shared memory: RB (mean, rstd)
// pairs, folded from the rows' G states in ws, or read from mean_in /
// rstd_in when those are given (a row's statistics computed beforehand).
// The CTAs of column block 0 write mean / rstd when given.  512
// threads rather than 256: twice the warps fold the rows' states at the
// CTA's start (16 x 1M bf16: 0.50 -> 0.54 of the copy bandwidth).
constexpr int kLnThreads = 512;
constexpr int kLnWarps = kLnThreads / 32;
template <class In>
__global__ void __launch_bounds__(kLnThreads, 2)
k_rowgrid_ln_out(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, int G, int RB,
                 float eps, const uint4 *__restrict__ ws, const float *__restrict__ mean_in,
                 const float *__restrict__ rstd_in, const float *__restrict__ gamma,
                 const float *__restrict__ beta, uint16_t *__restrict__ ybf,
                 float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  extern __shared__ float2 rowst[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r0 = (int64_t)blockIdx.y * RB;
  const int nr = (int)(rows - r0 < RB ? rows - r0 : RB);
  const int64_t u = (int64_t)blockIdx.x * kLnThreads + tid;
  const bool live = u < (cols >> 3);
  // gamma / beta of the thread's unit go out before the wait for the rows'
  // statistics
  float gv[8], bv[8];
  if (live) load_gamma_beta<8>(gamma, beta, u * 8, aligned32(gamma, beta), gv, bv);
  if (mean_in) {
    for (int j = tid; j < nr; j += kLnThreads) rowst[j] = make_float2(mean_in[r0 + j], rstd_in[r0 + j]);
  }
  for (int j = warp; !mean_in && j < nr; j += kLnWarps) {
    const Chan c = fold_row_chan(ws, r0 + j, G);
    if (lane == 0) {
      const float rs = rstd_of(c, cols, eps);
      rowst[j] = make_float2(c.mean, rs);
      if (blockIdx.x == 0) {
        if (mean) mean[r0 + j] = c.mean;
        if (rstd) rstd[r0 + j] = rs;
      }
    }
  }
  __syncthreads();
  if (!live) return;
  uint64_t g2[4], b2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    g2[q] = f2_pack(gv[2 * q], gv[2 * q + 1]);
    b2[q] = f2_pack(bv[2 * q], bv[2 * q + 1]);
  }
  const uint4 *xq = reinterpret_cast<const uint4 *>(x + r0 * cols);
  uint4 *yq = reinterpret_cast<uint4 *>(ybf + r0 * cols);
  const int64_t rw = cols / In::EPV;  // 16-byte words per row of x (per row of y: cols / 8)
  auto emit = [&](const GridUnit<In> &un, int j) {
    const float2 ms = rowst[j];
    const uint64_t mu2 = f2_pack(ms.x, ms.x), rs2 = f2_pack(ms.y, ms.y);
    uint64_t e2[4];
    un.pairs(e2);
    uint32_t pk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // fmaf((x - mu) * rs, gamma, beta), two elements at a time
      float lo, hi;
      f2_unpack(f2_fma(f2_mul(f2_sub(e2[k], mu2), rs2), g2[k], b2[k]), lo, hi);
      pk[k] = bf16x2_bits(lo, hi);
    }
    yq[(size_t)j * (size_t)(cols >> 3) + u] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  };
  const uint64_t pol = l2_evict_first_policy();  // x's last read
  // rows in flight a thread (fp32 units are twice the registers)
  constexpr int RU = In::EPV == 8 ? 6 : 2;
  int j0 = 0;
  for (; j0 + RU <= nr; j0 += RU) {
    GridUnit<In> un[RU];
#pragma unroll
    for (int k = 0; k < RU; ++k) un[k].load(xq + (size_t)(j0 + k) * rw, (int)u, pol);
#pragma unroll
    for (int k = 0; k < RU; ++k) emit(un[k], j0 + k);
  }
  if (j0 < nr) {
    GridUnit<In> un[RU];
#pragma unroll
    for (int k = 0; k < RU; ++k)
      if (j0 + k < nr) un[k].load(xq + (size_t)(j0 + k) * rw, (int)u, pol);
#pragma unroll
    for (int k = 0; k < RU; ++k)
      if (j0 + k < nr) emit(un[k], j0 + k);
  }
}

// The statistics alone: a warp per row.
__global__ void __launch_bounds__(kGridThreads)
k_rowgrid_stats_fin(int64_t rows, int64_t cols, int G, float eps, const uint4 *__restrict__ ws,
                    float *__restrict__ mean, float *__restrict__ rstd) {
  pdl_begin();
  const int64_t row = (int64_t)blockIdx.x * kGridWarps + (threadIdx.x >> 5);
  if (row >= rows) return;  // warp-uniform
  const Chan c = fold_row_chan(ws, row, G);
  if ((threadIdx.x & 31) == 0) {
    mean[row] = c.mean;
    rstd[row] = rstd_of(c, cols, eps);
  }
}

// The rewrite launch: column blocks of kLnThreads units, row groups of RB
// rows, at most one wave of 2 CTAs per SM.
template <class In>
int launch_ln_out(const typename In::S *x, int64_t rows, int64_t cols, int G, float eps,
                  const uint4 *ws, const float *mean_in, const float *rstd_in, const float *gamma,
                  const float *beta, uint16_t *ybf, float *mean, float *rstd, cudaStream_t s,
                  const DevInfo &d) {
  const int64_t cb = ((cols >> 3) + kLnThreads - 1) / kLnThreads;
  const int64_t want = (int64_t)2 * d.sm_count;
  int64_t groups = want / cb;
  if (groups > rows) groups = rows;
  if (groups < 1) groups = 1;
  int64_t RB = (rows + groups - 1) / groups;
  if (RB < (rows + 65534) / 65535) RB = (rows + 65534) / 65535;
  if (RB * (int64_t)sizeof(float2) > 48 * 1024) return RR_ERR_INVALID;
  groups = (rows + RB - 1) / RB;
  return cuda_status(launch_kernel(k_rowgrid_ln_out<In>, dim3((unsigned)cb, (unsigned)groups),
                                   dim3(kLnThreads), (size_t)RB * sizeof(float2), s, 0, x, rows,
                                   cols, G, (int)RB, eps, ws, mean_in, rstd_in, gamma, beta, ybf,
                                   mean, rstd));
}

template <class In>
int launch_grid(int mode, const void *xv, int64_t rows, int64_t cols, float eps, float *y,
                float *mean, float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
                int G, uint4 *ws, cudaStream_t s, const DevInfo &d) {
  using S = typename In::S;
  const S *x = (const S *)xv;
  const int64_t chunk = ((cols + G - 1) / G + 7) & ~int64_t(7);
  const unsigned nblk = (unsigned)(rows * G);
  if (log_enabled())
    std::fprintf(stderr, "rr: %s grid rows=%lld cols=%lld G=%d\n",
                 mode == kModeSoftmax ? "softmax" : (mode == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, G);
  cudaError_t e;
  if (mode == kModeSoftmax) {
    e = launch_kernel(k_rowgrid_part<In, kModeSoftmax, true>, dim3(nblk), dim3(kGridThreads), 0,
                      s, 0, x, cols, G, chunk, ws);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(launch_kernel(k_rowgrid_softmax_out<In>, dim3(nblk), dim3(kGridThreads), 0,
                                     s, 0, x, cols, G, chunk, (const uint4 *)ws, y));
  }
  e = launch_kernel(mode == kModeStats ? k_rowgrid_part<In, kModeStats, false>
                                        : k_rowgrid_part<In, kModeStats, true>,
                    dim3(nblk), dim3(kGridThreads), 0, s, 0, x, cols, G, chunk, ws);
  if (e != cudaSuccess) return cuda_status(e);
  if (mode == kModeStats)
    return cuda_status(launch_kernel(k_rowgrid_stats_fin,
                                     dim3((unsigned)((rows + kGridWarps - 1) / kGridWarps)),
                                     dim3(kGridThreads), 0, s, 0, rows, cols, G, eps,
                                     (const uint4 *)ws, mean, rstd));
  return launch_ln_out<In>(x, rows, cols, G, eps, ws, nullptr, nullptr, gamma, beta, ybf, mean,
                           rstd, s, d);
}

}  // namespace

int rowgrid_splits(int64_t rows, int64_t cols, int sm_count) {
  if (rows < 1 || cols < 8) return 1;
  int64_t g = (int64_t)kGridCtasPerSm * sm_count / rows;  // one wave
  const int64_t gmax = cols / kRowGridMinSlice;  // slices of at least this many elements
  if (g > gmax) g = gmax;
  if (g > kRowGridMaxSplits) g = kRowGridMaxSplits;
  if (g < 1) g = 1;
  // slices of fewer than 2^31 units
  const int64_t gmin = (cols + (int64_t(1) << 33) - 1) >> 33;
  return (int)(g < gmin ? gmin : g);
}

int launch_rowgrid(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols, float eps,
                   float *y, float *mean, float *rstd, const float *gamma, const float *beta,
                   uint16_t *ybf, int G, void *ws, size_t ws_bytes, cudaStream_t s,
                   const DevInfo &d) {
  if (G < 1 || G > kRowGridMaxSplits || cols % 8 != 0 || (uintptr_t)x % 16 != 0 || !ws ||
      (uintptr_t)ws % 16 != 0)
    return RR_ERR_INVALID;
  if (rows * G > INT_MAX || rowgrid_ws_bytes(rows, G) > ws_bytes) return RR_ERR_INVALID;
  // a slice's 8-element units and a row's units are counted in an int
  if (((cols + G - 1) / G + 7) / 8 > INT_MAX || cols / 8 > INT_MAX) return RR_ERR_INVALID;
  if (mode == kModeSoftmax && (uintptr_t)y % 32 != 0) return RR_ERR_INVALID;
  if (mode == kModeLayernorm &&
      ((uintptr_t)ybf % 16 != 0 || (uintptr_t)gamma % 16 != 0 || (uintptr_t)beta % 16 != 0))
    return RR_ERR_INVALID;
  if (in_dtype == RR_BF16)
    return launch_grid<InBF16>(mode, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, G,
                               (uint4 *)ws, s, d);
  return launch_grid<InF32>(mode, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, G,
                            (uint4 *)ws, s, d);
}

int launch_ln_apply(int in_dtype, const void *x, int64_t rows, int64_t cols, const float *mean_in,
                    const float *rstd_in, const float *gamma, const float *beta, uint16_t *ybf,
                    cudaStream_t s, const DevInfo &d) {
  if (cols % 8 != 0 || cols / 8 > INT_MAX || (uintptr_t)x % 16 != 0 || !mean_in || !rstd_in ||
      (uintptr_t)ybf % 16 != 0 || (uintptr_t)gamma % 16 != 0 || (uintptr_t)beta % 16 != 0)
    return RR_ERR_INVALID;
  if (rows == 0 || cols == 0) return RR_OK;
  if (log_enabled())
    std::fprintf(stderr, "rr: layernorm apply rows=%lld cols=%lld\n", (long long)rows,
                 (long long)cols);
  if (in_dtype == RR_BF16)
    return launch_ln_out<InBF16>((const InBF16::S *)x, rows, cols, 0, 0.0f, nullptr, mean_in,
                                 rstd_in, gamma, beta, ybf, nullptr, nullptr, s, d);
  return launch_ln_out<InF32>((const InF32::S *)x, rows, cols, 0, 0.0f, nullptr, mean_in, rstd_in,
                              gamma, beta, ybf, nullptr, nullptr, s, d);
}

}  // namespace rr
