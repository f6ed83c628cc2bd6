// rowstaged.cu -- the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise: softmax, layernorm statistics, layernorm rewrite)
// for rows too long to hold in a CTA's registers, with the row staged in
// shared memory so that HBM is read once.
//
// A cluster of C CTAs per row (C = 1: a CTA per row); CTA r owns the slice
// [r * chunk, min((r + 1) * chunk, cols)) with chunk a multiple of 8
// elements, so every slice starts 16-byte aligned when the row does.  One
// thread copies the slice into the CTA's shared memory with 1-D bulk copies
// (the copy engine; completion counted on an mbarrier), and every pass then
// reads shared memory:
//   softmax:   slice max -> block max -> cluster max M ("cluster_allreduce"
//              page, rank-order fold); slice sum of e^(x - M) -> block sum ->
//              cluster sum S; write y = e^(x - M) / S.
//   layernorm: slice sum -> mean; slice sum of (x - mean)^2 -> variance ->
//              rstd; the rewrite bf16((x - mean) * rstd * gamma + beta).
// The two combines of a row use two slots without a tail sync and the CTA
// ends with one cluster barrier, as the split-K tier does.  Every CTA of a
// cluster folds the same partials in rank order, so all hold the same
// statistics.  A slice of up to kStageMaxBytes leaves room for two CTAs on
// an SM, which overlap one's copy with the other's passes; within a CTA the
// first pass folds the slice piece by piece as the pieces land.  (A
// persistent form with two stage buffers per CTA, one CTA per SM, measured
// slower: 8 warps could not keep up with the passes over shared memory.)
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"
#include "rowwise.cuh"

namespace rr {
namespace {

#ifndef RR_STAGE_THREADS
#define RR_STAGE_THREADS 256
#endif
constexpr int kStageThreads = RR_STAGE_THREADS;

// Unpacks the 8 elements of vector v of a staged slice.
template <class In>
__device__ __forceinline__ void staged8(const unsigned char *stage, int v, float (&e)[8]) {
  if constexpr (In::EPV == 8) {
    In::unpack(*reinterpret_cast<const uint4 *>(stage + (size_t)v * 16), e);
  } else {
    const uint4 a = *reinterpret_cast<const uint4 *>(stage + (size_t)v * 32);
    const uint4 b = *reinterpret_cast<const uint4 *>(stage + (size_t)v * 32 + 16);
    e[0] = __uint_as_float(a.x); e[1] = __uint_as_float(a.y);
    e[2] = __uint_as_float(a.z); e[3] = __uint_as_float(a.w);
    e[4] = __uint_as_float(b.x); e[5] = __uint_as_float(b.y);
    e[6] = __uint_as_float(b.z); e[7] = __uint_as_float(b.w);
  }
}
// Element i of a staged slice.
template <class In>
__device__ __forceinline__ float staged1(const unsigned char *stage, int i) {
  if constexpr (In::EPV == 8) {
    return __uint_as_float(((uint32_t) reinterpret_cast<const uint16_t *>(stage)[i]) << 16);
  } else {
    return reinterpret_cast<const float *>(stage)[i];
  }
}

// The slice arrives in pieces of kPiece bytes, each counted on its own
// mbarrier, so that the first pass folds a piece as soon as it lands while
// the copy engine still writes the next ones.
constexpr uint32_t kPiece = 16384;
constexpr int kMaxPieces = (int)((kStageMaxBytes + kPiece - 1) / kPiece);

// Visits the vectors (8 elements each) of a staged slice for the first pass,
// piece by piece in arrival order, then the tail elements: f(e[8]) for each
// whole vector, f1(x) for each tail element.  Returns false if a wait gave
// up.
template <class In, int T, class F, class F1>
__device__ __forceinline__ bool first_pass(const unsigned char *stage, uint64_t *full, int npieces,
                                           int nv, int n, volatile int *dead, F f, F1 f1) {
  constexpr int kVecBytes = 8 * (int)sizeof(typename In::S);
  constexpr int kVecPerPiece = (int)kPiece / kVecBytes;
  bool ok = true;
  for (int p = 0; p < npieces; ++p) {
    if (!mbar_wait_or_die(&full[p], 0, kWaitBudget, dead, false)) ok = false;
    const int end = (p + 1) * kVecPerPiece < nv ? (p + 1) * kVecPerPiece : nv;
    for (int v = p * kVecPerPiece + (int)threadIdx.x; v < end; v += T) {
      float e[8];
      staged8<In>(stage, v, e);
      f(e);
    }
  }
  for (int i = nv * 8 + (int)threadIdx.x; i < n; i += T) f1(staged1<In>(stage, i));
  return ok;
}

// MODE kModeSoftmax: y (fp32); kModeStats: mean, rstd; kModeLayernorm: ybf
// (bf16), mean / rstd optional.  Requires x rows 16-byte aligned (x 16-byte
// aligned, cols a multiple of the 16-byte vector), chunk a multiple of 8 and
// chunk * sizeof(element) <= kStageMaxBytes bytes of dynamic shared memory.
template <class In, int MODE>
__global__ void __launch_bounds__(kStageThreads)
k_rowwise_staged(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, int chunk,
                 float eps, float *__restrict__ y, float *__restrict__ mean,
                 float *__restrict__ rstd, const float *__restrict__ gamma,
                 const float *__restrict__ beta, uint16_t *__restrict__ ybf, int *err) {
  pdl_begin();
  constexpr int T = kStageThreads;
  extern __shared__ __align__(128) unsigned char stage[];
  __shared__ __align__(8) uint64_t full[kMaxPieces];
  __shared__ float red[2][T / 32];
  __shared__ float slot[2][2];
  __shared__ int dead;
  const int tid = threadIdx.x;
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t row = cluster_id_x();
  const int64_t b0 = (int64_t)r * chunk < cols ? (int64_t)r * chunk : cols;
  const int64_t b1 = b0 + chunk < cols ? b0 + chunk : cols;
  const int n = (int)(b1 - b0);   // elements of this CTA's slice
  const int nv = n >> 3;          // whole 8-element vectors; the rest is a tail
  const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(typename In::S);  // a multiple of 16
  const int npieces = (int)((bytes + kPiece - 1) / kPiece);

  if (tid == 0) {
    dead = 0;
    for (int p = 0; p < npieces; ++p) mbar_init(&full[p], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const unsigned char *src = reinterpret_cast<const unsigned char *>(x + row * cols + b0);
    for (int p = 0; p < npieces; ++p) {
      const uint32_t off = (uint32_t)p * kPiece;
      const uint32_t len = bytes - off < kPiece ? bytes - off : kPiece;
      mbar_arrive_expect_tx(&full[p], len);
      bulk_g2s(stage + off, src + off, len, &full[p]);
    }
  }

  if constexpr (MODE == kModeSoftmax) {
    float m = -INFINITY;
    if (!first_pass<In, T>(stage, full, npieces, nv, n, &dead,
                           [&](const float (&e)[8]) {
#pragma unroll
                             for (int j = 0; j < 8; ++j) m = fmaxf(m, e[j]);
                           },
                           [&](float v) { m = fmaxf(m, v); }))
      set_error(err, kErrTimeout);
    m = block_reduce<MaxF32, T>(m, red[0]);
    float v1[1] = {m}, M[1];
    cluster_allreduce<MaxF32, 1>(slot[0], v1, C, /*tail_sync=*/false, M);  // combine 1
    const float Mx = M[0];
    const float mb = Mx * kLog2e;
    float s = 0.0f;
    if (Mx != -INFINITY) {
      for (int v = tid; v < nv; v += T) {
        float e[8];
        staged8<In>(stage, v, e);
#pragma unroll
        for (int j = 0; j < 8; ++j) s += ex2_approx(fmaf(e[j], kLog2e, -mb));
      }
      for (int i = nv * 8 + tid; i < n; i += T)
        s += ex2_approx(fmaf(staged1<In>(stage, i), kLog2e, -mb));
    }
    s = block_reduce<SumF32, T>(s, red[1]);
    float v2[1] = {s}, Ssum[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, Ssum);  // combine 2
    const float inv = 1.0f / Ssum[0];
    float *yr = y + row * cols + b0;
    for (int v = tid; v < nv; v += T) {
      float e[8];
      staged8<In>(stage, v, e);
      float o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o[j] = (Mx == -INFINITY) ? 0.0f : ex2_approx(fmaf(e[j], kLog2e, -mb)) * inv;
      if constexpr (In::EPV == 8) {
        st_stream_v8(yr + (int64_t)v * 8, o);
      } else {
        st_stream_v4(yr + (int64_t)v * 8, o[0], o[1], o[2], o[3]);
        st_stream_v4(yr + (int64_t)v * 8 + 4, o[4], o[5], o[6], o[7]);
      }
    }
    for (int i = nv * 8 + tid; i < n; i += T)
      yr[i] = (Mx == -INFINITY) ? 0.0f
                                : ex2_approx(fmaf(staged1<In>(stage, i), kLog2e, -mb)) * inv;
  } else {
    float a = 0.0f;
    if (!first_pass<In, T>(stage, full, npieces, nv, n, &dead,
                           [&](const float (&e)[8]) {
#pragma unroll
                             for (int j = 0; j < 8; ++j) a += e[j];
                           },
                           [&](float v) { a += v; }))
      set_error(err, kErrTimeout);
    a = block_reduce<SumF32, T>(a, red[0]);
    float v1[1] = {a}, tot[1];
    cluster_allreduce<SumF32, 1>(slot[0], v1, C, /*tail_sync=*/false, tot);  // combine 1
    const float mu = tot[0] / (float)cols;
    float q = 0.0f;
    for (int v = tid; v < nv; v += T) {
      float e[8];
      staged8<In>(stage, v, e);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float dl = e[j] - mu;
        q = fmaf(dl, dl, q);
      }
    }
    for (int i = nv * 8 + tid; i < n; i += T) {
      const float dl = staged1<In>(stage, i) - mu;
      q = fmaf(dl, dl, q);
    }
    q = block_reduce<SumF32, T>(q, red[1]);
    float v2[1] = {q}, tq[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, tq);  // combine 2
    const float rs = 1.0f / sqrtf(tq[0] / (float)cols + eps);
    if (r == 0 && tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
    if constexpr (MODE == kModeLayernorm) {
      uint16_t *yr = ybf + row * cols + b0;
      const bool gb32 = aligned32(gamma + b0, beta + b0);
      for (int v = tid; v < nv; v += T) {
        float e[8], g[8], bt[8];
        staged8<In>(stage, v, e);
        load_gamma_beta<8>(gamma + b0, beta + b0, (int64_t)v * 8, gb32, g, bt);
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2)
          pk[j / 2] = bf16x2_bits(fmaf((e[j] - mu) * rs, g[j], bt[j]),
                                  fmaf((e[j + 1] - mu) * rs, g[j + 1], bt[j + 1]));
        if constexpr (In::EPV == 8) {
          *reinterpret_cast<uint4 *>(yr + (int64_t)v * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        } else {
          *reinterpret_cast<uint2 *>(yr + (int64_t)v * 8) = make_uint2(pk[0], pk[1]);
          *reinterpret_cast<uint2 *>(yr + (int64_t)v * 8 + 4) = make_uint2(pk[2], pk[3]);
        }
      }
      for (int i = nv * 8 + tid; i < n; i += T) {
        const __nv_bfloat16 h = __float2bfloat16_rn(fmaf(
            (staged1<In>(stage, i) - mu) * rs, __ldg(gamma + b0 + i), __ldg(beta + b0 + i)));
        yr[i] = *reinterpret_cast<const uint16_t *>(&h);
      }
    }
  }
  if (C > 1) cluster_sync();  // no CTA leaves while a peer may read its slots
}

// 8 consecutive floats from p, which lies `sh` floats (0..3) past a 16-byte
// boundary: two or three aligned 16-byte loads and a selection fixed by sh
// (uniform over the CTA).  The caller checks that the aligned window
// [p - sh, p - sh + 8 or 12) lies inside the array.
__device__ __forceinline__ void load8_shifted(const float *p, int sh, float (&o)[8]) {
  const float4 *q = reinterpret_cast<const float4 *>(p - sh);
  const float4 a = __ldg(q), b = __ldg(q + 1);
  if (sh == 0) {
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    return;
  }
  const float4 c = __ldg(q + 2);
  if (sh == 1) {
    o[0] = a.y; o[1] = a.z; o[2] = a.w; o[3] = b.x; o[4] = b.y; o[5] = b.z; o[6] = b.w; o[7] = c.x;
  } else if (sh == 2) {
    o[0] = a.z; o[1] = a.w; o[2] = b.x; o[3] = b.y; o[4] = b.z; o[5] = b.w; o[6] = c.x; o[7] = c.y;
  } else {
    o[0] = a.w; o[1] = b.x; o[2] = b.y; o[3] = b.z; o[4] = b.w; o[5] = c.x; o[6] = c.y; o[7] = c.z;
  }
}

// ---------------------------------------------------------------------------
// Staged rows that do not start 16-byte aligned (a width that is not a
// multiple of the 16-byte vector, or a misaligned x): the same passes over
// a slice copied into shared memory at its address's offset within its
// 16-byte chunk, so that smem byte k holds global byte floor16(slice) + k.
// The slice's whole 16-byte chunks come by bulk copies; the elements of its
// partial first and last chunks by plain loads.  Every pass walks the
// 8-element vectors of that image, vector v holding slice elements
// 8v + j - hoff (hoff = the slice's element offset in its first chunk), and
// leaves the slots outside [0, n) of the first and last vector out of the
// fold.  Outputs go as vectors where the output row's shifted base is
// aligned, else element by element; gamma and beta are read element by
// element (their offset varies with the row).
// ---------------------------------------------------------------------------
template <class In, int MODE>
__global__ void __launch_bounds__(kStageThreads)
k_rowwise_staged_mis(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, int chunk,
                     float eps, float *__restrict__ y, float *__restrict__ mean,
                     float *__restrict__ rstd, const float *__restrict__ gamma,
                     const float *__restrict__ beta, uint16_t *__restrict__ ybf, int *err) {
  pdl_begin();
  using S = typename In::S;
  constexpr int T = kStageThreads;
  constexpr int E = (int)sizeof(S);
  extern __shared__ __align__(128) unsigned char stage[];
  __shared__ __align__(8) uint64_t full;
  __shared__ float red[2][T / 32];
  __shared__ float slot[2][2];
  __shared__ int dead;
  const int tid = threadIdx.x;
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t row = cluster_id_x();
  const int64_t b0 = (int64_t)r * chunk < cols ? (int64_t)r * chunk : cols;
  const int64_t b1 = b0 + chunk < cols ? b0 + chunk : cols;
  const int n = (int)(b1 - b0);
  const S *ps = x + row * cols + b0;
  const int hoffB = (int)((uintptr_t)ps & 15u);      // bytes before the slice in its chunk
  const int hoff = hoffB / E;
  const unsigned char *base = reinterpret_cast<const unsigned char *>(ps) - hoffB;
  const int span = hoffB + n * E;                    // bytes of the image
  const int nch = (span + 15) >> 4;                  // 16-byte chunks
  const int c_lo = hoffB ? 1 : 0;                    // whole chunks [c_lo, c_hi)
  const int c_hi = (span & 15) ? nch - 1 : nch;
  const int head_n = c_lo ? ((16 - hoffB) / E < n ? (16 - hoffB) / E : n) : 0;
  int tail_0 = n;                                    // elements of a partial last chunk
  if ((span & 15) && nch - 1 >= c_lo) {
    const int t0 = (16 * (nch - 1) - hoffB) / E;
    tail_0 = t0 > head_n ? t0 : head_n;
  }
  const int nvt = (hoff + n + 7) >> 3;               // 8-element vectors of the image

  if (tid == 0) {
    dead = 0;
    mbar_init(&full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = c_hi > c_lo ? (uint32_t)(c_hi - c_lo) * 16u : 0u;
    mbar_arrive_expect_tx(&full, bytes);
    for (uint32_t off = 0; off < bytes; off += kPiece)
      bulk_g2s(stage + 16 * c_lo + off, base + 16 * c_lo + off,
               bytes - off < kPiece ? bytes - off : kPiece, &full);
  }
  S *se = reinterpret_cast<S *>(stage);
  for (int i = tid; i < head_n; i += T) se[hoff + i] = ps[i];
  for (int i = tail_0 + tid; i < n; i += T) se[hoff + i] = ps[i];
  if (!mbar_wait_or_die(&full, 0, kWaitBudget, &dead, false)) set_error(err, kErrTimeout);
  __syncthreads();  // the plain stores of the edge elements

  // fold of vector v: f(e, valid) for each slot; edge vectors mask
  auto visit = [&](int v, auto f) {
    float e[8];
    staged8<In>(stage, v, e);
    if (v == 0 || v == nvt - 1) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = 8 * v + j - hoff;
        f(j, e[j], i >= 0 && i < n);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) f(j, e[j], true);
    }
  };

  if constexpr (MODE == kModeSoftmax) {
    float m = -INFINITY;
    for (int v = tid; v < nvt; v += T)
      visit(v, [&](int, float e, bool ok) { m = ok ? fmaxf(m, e) : m; });
    m = block_reduce<MaxF32, T>(m, red[0]);
    float v1[1] = {m}, M[1];
    cluster_allreduce<MaxF32, 1>(slot[0], v1, C, /*tail_sync=*/false, M);  // combine 1
    const float Mx = M[0];
    const float mb = Mx * kLog2e;
    float s = 0.0f;
    if (Mx != -INFINITY) {
      for (int v = tid; v < nvt; v += T)
        visit(v, [&](int, float e, bool ok) {
          if (ok) s += ex2_approx(fmaf(e, kLog2e, -mb));
        });
    }
    s = block_reduce<SumF32, T>(s, red[1]);
    float v2[1] = {s}, Ssum[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, Ssum);  // combine 2
    const float inv = 1.0f / Ssum[0];
    float *yv = y + row * cols + b0 - hoff;          // element i of the slice at yv[hoff + i]
    const bool vy = ((uintptr_t)yv % (In::EPV == 8 ? 32 : 16)) == 0;
    for (int v = tid; v < nvt; v += T) {
      float e[8];
      staged8<In>(stage, v, e);
      float o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o[j] = (Mx == -INFINITY) ? 0.0f : ex2_approx(fmaf(e[j], kLog2e, -mb)) * inv;
      if (vy && v != 0 && v != nvt - 1) {
        if constexpr (In::EPV == 8) {
          st_stream_v8(yv + (int64_t)v * 8, o);
        } else {
          st_stream_v4(yv + (int64_t)v * 8, o[0], o[1], o[2], o[3]);
          st_stream_v4(yv + (int64_t)v * 8 + 4, o[4], o[5], o[6], o[7]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = 8 * v + j - hoff;
          if (i >= 0 && i < n) yv[hoff + i] = o[j];
        }
      }
    }
  } else {
    float a = 0.0f;
    for (int v = tid; v < nvt; v += T)
      visit(v, [&](int, float e, bool ok) { a += ok ? e : 0.0f; });
    a = block_reduce<SumF32, T>(a, red[0]);
    float v1[1] = {a}, tot[1];
    cluster_allreduce<SumF32, 1>(slot[0], v1, C, /*tail_sync=*/false, tot);  // combine 1
    const float mu = tot[0] / (float)cols;
    float q = 0.0f;
    for (int v = tid; v < nvt; v += T)
      visit(v, [&](int, float e, bool ok) {
        const float dl = e - mu;
        q = ok ? fmaf(dl, dl, q) : q;
      });
    q = block_reduce<SumF32, T>(q, red[1]);
    float v2[1] = {q}, tq[1];
    cluster_allreduce<SumF32, 1>(slot[1], v2, C, /*tail_sync=*/false, tq);  // combine 2
    const float rs = 1.0f / sqrtf(tq[0] / (float)cols + eps);
    if (r == 0 && tid == 0) {
      if (mean) mean[row] = mu;
      if (rstd) rstd[row] = rs;
    }
    if constexpr (MODE == kModeLayernorm) {
      uint16_t *yv = ybf + row * cols + b0 - hoff;
      const float *gv = gamma + b0 - hoff, *bv = beta + b0 - hoff;
      const bool vy = ((uintptr_t)yv % 16) == 0;
      const int gsh = (int)(((uintptr_t)gv >> 2) & 3u), bsh = (int)(((uintptr_t)bv >> 2) & 3u);
      for (int v = tid; v < nvt; v += T) {
        float e[8];
        staged8<In>(stage, v, e);
        const bool edge = v == 0 || v == nvt - 1;
        float o[8];
        // gamma / beta as shifted vectors where every slot is in the row and
        // both aligned windows lie inside [0, cols)
        const int64_t g0 = b0 - hoff + 8 * (int64_t)v;
        const bool gin = g0 - gsh >= 0 && g0 - gsh + (gsh ? 12 : 8) <= cols &&
                         g0 - bsh >= 0 && g0 - bsh + (bsh ? 12 : 8) <= cols;
        if (!edge && gin) {
          float g[8], bt[8];
          load8_shifted(gv + 8 * v, gsh, g);
          load8_shifted(bv + 8 * v, bsh, bt);
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = fmaf((e[j] - mu) * rs, g[j], bt[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = 8 * v + j - hoff;
            const bool ok = i >= 0 && i < n;
            o[j] = ok ? fmaf((e[j] - mu) * rs, __ldg(gv + 8 * v + j), __ldg(bv + 8 * v + j)) : 0.0f;
          }
        }
        if (vy && !edge) {
          *reinterpret_cast<uint4 *>(yv + (int64_t)v * 8) =
              make_uint4(bf16x2_bits(o[0], o[1]), bf16x2_bits(o[2], o[3]), bf16x2_bits(o[4], o[5]),
                         bf16x2_bits(o[6], o[7]));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = 8 * v + j - hoff;
            if (i >= 0 && i < n) {
              const __nv_bfloat16 h = __float2bfloat16_rn(o[j]);
              yv[hoff + i] = *reinterpret_cast<const uint16_t *>(&h);
            }
          }
        }
      }
    }
  }
  if (C > 1) cluster_sync();  // no CTA leaves while a peer may read its slots
}

template <class In, int MODE>
int launch_mode(const void *x, int64_t rows, int64_t cols, float eps, float *y, float *mean,
                float *rstd, const float *gamma, const float *beta, uint16_t *ybf, int C,
                bool aligned, cudaStream_t s, const DevInfo &d) {
  // every operand aligned for the vector forms: the plain kernel; otherwise
  // the misaligned one, whose image is up to 8 elements longer than a slice
  auto kern = aligned ? k_rowwise_staged<In, MODE> : k_rowwise_staged_mis<In, MODE>;
  const int64_t chunk = rowwise_staged_chunk(cols, C);
  const size_t smem = (size_t)(chunk + (aligned ? 0 : 8)) * sizeof(typename In::S);
  if (chunk < 0 || smem > (size_t)kStageMaxBytes) return RR_ERR_INVALID;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kStageMaxBytes);
  if (e != cudaSuccess) return cuda_status(e);
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (occupancy_clusters((const void *)kern, kStageThreads, smem, C, d.device) < 1)
    return RR_ERR_UNSUPPORTED;
  if (rows * C > 0x7fffffffLL) return RR_ERR_INVALID;
  if (log_enabled())
    std::fprintf(stderr, "rr: %s staged%s rows=%lld cols=%lld C=%d chunk=%lld smem=%zu\n",
                 MODE == kModeSoftmax ? "softmax" : (MODE == kModeStats ? "lnstats" : "layernorm"),
                 aligned ? "" : " (misaligned rows)", (long long)rows, (long long)cols, C,
                 (long long)chunk, smem);
  return cuda_status(launch_kernel(kern, dim3((unsigned)(rows * C)), dim3(kStageThreads), smem, s,
                                   C, (const typename In::S *)x, rows, cols, (int)chunk, eps, y,
                                   mean, rstd, gamma, beta, ybf, d.err_word));
}

}  // namespace

int64_t rowwise_staged_chunk(int64_t cols, int C) {
  if (C < 1 || cols < 1) return -1;
  return ((cols + C - 1) / C + 7) & ~int64_t(7);
}

int rowwise_staged_cluster(int64_t cols, int in_dtype, int max_cluster, bool aligned) {
  const int64_t elt = in_dtype == RR_BF16 ? 2 : 4;
  for (int C = 1; C <= 16 && C <= max_cluster; C *= 2)
    if ((rowwise_staged_chunk(cols, C) + (aligned ? 0 : 8)) * elt <= kStageMaxBytes) return C;
  return 0;
}

int launch_rowwise_staged(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                          float eps, float *y, float *mean, float *rstd, const float *gamma,
                          const float *beta, uint16_t *ybf, int C, bool aligned, cudaStream_t s,
                          const DevInfo &d) {
  if (in_dtype == RR_BF16) {
    switch (mode) {
      case kModeSoftmax: return launch_mode<InBF16, kModeSoftmax>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
      case kModeStats: return launch_mode<InBF16, kModeStats>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
      default: return launch_mode<InBF16, kModeLayernorm>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
    }
  }
  switch (mode) {
    case kModeSoftmax: return launch_mode<InF32, kModeSoftmax>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
    case kModeStats: return launch_mode<InF32, kModeStats>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
    default: return launch_mode<InF32, kModeLayernorm>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, aligned, s, d);
  }
}

}  // namespace rr
