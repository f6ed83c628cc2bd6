// rowwarp.cu -- warp tier of the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise, tier semantics: a warp per row for rows too short
// to keep a CTA busy): softmax, layernorm statistics and the layernorm
// rewrite for rows of up to 256 16-byte vectors (2048 bf16 / 1024 fp32
// elements) when there are many of them.
//
// A segment of L lanes of a warp owns a row (32 / L rows per warp at a
// time; L = 1 is a thread per row) and holds it in registers: lane `sub` of
// the segment holds vectors k * L + sub, k < NV, so each load instruction of
// the segment covers L * 16 contiguous bytes.  Both reductions of a row are
// xor butterflies inside the segment -- no shared memory and no barrier --
// and the next row's raw vectors are loaded before the current row is
// reduced and written, so a lane keeps up to 2 * NV 16-byte loads in flight.
// Vector indices past the row end are clamped to the row's last vector
// (loaded, then left out of every fold); a segment past the last row
// re-reads the last row and writes nothing.  So every load is unconditional
// and every lane takes part in every shuffle.
//
// Rows that are not aligned 16-byte vectors (a width that is not a multiple
// of 8 bf16 / 4 fp32 elements, or a misaligned base) take a chunked form --
// the row's whole aligned 16-byte chunks spread over the segment like the
// vectors, its head and tail elements held one by one -- or, for outputs
// that do not sit at x's offset within a chunk and for the rewrite's
// narrowest rows, an element-wise form.
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"
#include "rowwise.cuh"

namespace rr {
namespace {

constexpr int kWarpRowMaxThreads = 256;

// MODE kModeSoftmax: y (fp32) = e^(x - M) / S with (M, S) the row's (max,
// sum) pair; kModeStats: mean, rstd; kModeLayernorm: ybf (bf16) =
// (x - mean) * rstd * gamma + beta, mean / rstd optional.  The arithmetic
// per element is that of the block tier's register form; only the order in
// which the per-lane partials are combined differs (a butterfly over the L
// lanes instead of warp trees and a block fold).
template <class In, int MODE, int L, int NV>
__global__ void __launch_bounds__(kWarpRowMaxThreads)
k_rowwise_warp(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
               float *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd,
               const float *__restrict__ gamma, const float *__restrict__ beta,
               uint16_t *__restrict__ ybf) {
  pdl_begin();
  constexpr int EPV = In::EPV, RPW = 32 / L;
  const int lane = threadIdx.x & 31, seg = lane / L, sub = lane % L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = (((int64_t)gridDim.x * blockDim.x) >> 5) * RPW;
  const int nvec = cols / EPV;
  const bool gb32 = MODE == kModeLayernorm && aligned32(gamma, beta);
  uint4 raw[NV];
  auto fetch = [&](int64_t r) {
    const int64_t rc = r < rows ? r : rows - 1;
    const uint4 *q = reinterpret_cast<const uint4 *>(x + rc * (int64_t)cols);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int idx = k * L + sub;
      raw[k] = ld_stream_u4(q + (idx < nvec ? idx : nvec - 1));
    }
  };
  int64_t r0 = warp * RPW;
  if (r0 < rows) fetch(r0 + seg);
  for (; r0 < rows; r0 += stride) {  // warp-uniform trip count
    const int64_t row = r0 + seg;
    float v[NV][EPV];
#pragma unroll
    for (int k = 0; k < NV; ++k) In::unpack(raw[k], v[k]);
    if (r0 + stride < rows) fetch(r0 + stride + seg);
    if constexpr (MODE == kModeSoftmax) {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (k * L + sub < nvec) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) m = fmaxf(m, v[k][e]);
        }
      float s = 0.0f;
      if (m != -INFINITY) {
        const float mb = m * kLog2e;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          float sk = 0.0f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float p = ex2_approx(fmaf(v[k][e], kLog2e, -mb));
            v[k][e] = p;
            sk += p;
          }
          if (k * L + sub < nvec) s += sk;
        }
      } else {
        // every element the lane holds is -inf: e^(x - M) = 0, not -inf * 0
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
          for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
      }
      float M = m, S = s;
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1)
        ms_combine(M, S, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S, o));
      const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S);
      if (row < rows) {
        float *yr = y + row * (int64_t)cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const int idx = k * L + sub;
          if (idx < nvec) {
            if constexpr (EPV == 8) {
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
      }
    } else {
      // two elements per packed fp32 instruction (even and odd elements in
      // the two halves)
      uint64_t sa = 0;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (k * L + sub < nvec) {
#pragma unroll
          for (int e = 0; e < EPV; e += 2) sa = f2_add(sa, f2_pack(v[k][e], v[k][e + 1]));
        }
      float slo, shi;
      f2_unpack(sa, slo, shi);
      const float mu = warp_allreduce<SumF32, L>(slo + shi) / (float)cols;
      const uint64_t nmu2 = f2_pack(-mu, -mu);
      uint64_t qa = 0;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (k * L + sub < nvec) {
#pragma unroll
          for (int e = 0; e < EPV; e += 2) {
            const uint64_t d = f2_add(f2_pack(v[k][e], v[k][e + 1]), nmu2);
            qa = f2_fma(d, d, qa);
          }
        }
      float qlo, qhi;
      f2_unpack(qa, qlo, qhi);
      const float var = warp_allreduce<SumF32, L>(qlo + qhi) * (1.0f / (float)cols);
      const float rs = 1.0f / sqrtf(var + eps);
      if (row < rows) {
        if constexpr (MODE == kModeLayernorm) {
          uint16_t *yr = ybf + row * (int64_t)cols;
          const uint64_t mu2 = f2_pack(mu, mu), rs2 = f2_pack(rs, rs);
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            const int idx = k * L + sub;
            if (idx < nvec) {
              float g[EPV], b[EPV];
              load_gamma_beta<EPV>(gamma, beta, (int64_t)idx * EPV, gb32, g, b);
              uint32_t pk[EPV / 2];
#pragma unroll
              for (int e = 0; e < EPV; e += 2) {
                // fmaf((x - mu) * rs, gamma, beta), two elements at a time
                float lo, hi;
                f2_unpack(f2_fma(f2_mul(f2_sub(f2_pack(v[k][e], v[k][e + 1]), mu2), rs2),
                                 f2_pack(g[e], g[e + 1]), f2_pack(b[e], b[e + 1])), lo, hi);
                pk[e / 2] = bf16x2_bits(lo, hi);
              }
              if constexpr (EPV == 8) {
                *reinterpret_cast<uint4 *>(yr + idx * EPV) =
                    make_uint4(pk[0], pk[1 % (EPV / 2)], pk[2 % (EPV / 2)], pk[3 % (EPV / 2)]);
              } else {
                *reinterpret_cast<uint2 *>(yr + idx * EPV) = make_uint2(pk[0], pk[1 % (EPV / 2)]);
              }
            }
          }
        }
        if (sub == 0) {
          if (mean) mean[row] = mu;
          if (rstd) rstd[row] = rs;
        }
      }
    }
  }
}

// Element-wise form, for rows that are not made of aligned 16-byte vectors
// (a width that is not a multiple of 8 bf16 / 4 fp32 elements, or a
// misaligned operand) of up to 32 * K elements: lane `sub` of a segment of L
// lanes holds elements k * L + sub, k < K (consecutive lanes read
// consecutive elements), with clamped, unconditional loads and the slots
// past the row's end left out of every fold.  Reductions, outputs and the
// per-element arithmetic as in the vector form; stores element by element.
// For softmax rows of 16 or more elements a lane, the next row's elements
// are loaded (as raw bf16 / fp32) before the current row is reduced and
// written (measured: a loss for shorter rows and for the rewrite).
template <class In, int MODE, int L, int K>
__global__ void __launch_bounds__(kWarpRowMaxThreads)
k_rowwise_warp_el(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
                  float *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd,
                  const float *__restrict__ gamma, const float *__restrict__ beta,
                  uint16_t *__restrict__ ybf) {
  pdl_begin();
  constexpr int RPW = 32 / L;
  const int lane = threadIdx.x & 31, seg = lane / L, sub = lane % L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = (((int64_t)gridDim.x * blockDim.x) >> 5) * RPW;
  typename In::S raw[K];
  auto fetch = [&](int64_t r) {
    const int64_t rc = r < rows ? r : rows - 1;
    const typename In::S *xr = x + rc * (int64_t)cols;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int i = k * L + sub;
      raw[k] = __ldg(xr + (i < cols ? i : cols - 1));
    }
  };
  constexpr bool PF = MODE == kModeSoftmax && K >= 16;
  int64_t r0 = warp * RPW;
  if constexpr (PF) {
    if (r0 < rows) fetch(r0 + seg);
  }
  for (; r0 < rows; r0 += stride) {  // warp-uniform trip count
    const int64_t row = r0 + seg;
    if constexpr (!PF) fetch(row);
    float v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = In::cvt(raw[k]);
    if constexpr (PF) {
      if (r0 + stride < rows) fetch(r0 + stride + seg);
    }
    if constexpr (MODE == kModeSoftmax) {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k * L + sub < cols) m = fmaxf(m, v[k]);
      float s = 0.0f;
      if (m != -INFINITY) {
        const float mb = m * kLog2e;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const float p = ex2_approx(fmaf(v[k], kLog2e, -mb));
          v[k] = p;
          if (k * L + sub < cols) s += p;
        }
      } else {
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] = 0.0f;
      }
      float M = m, S = s;
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1)
        ms_combine(M, S, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S, o));
      const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S);
      if (row < rows) {
        float *yr = y + row * (int64_t)cols;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int i = k * L + sub;
          if (i < cols) yr[i] = v[k] * f;
        }
      }
    } else {
      float s = 0.0f;
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k * L + sub < cols) s += v[k];
      const float mu = warp_allreduce<SumF32, L>(s) / (float)cols;
      float qs = 0.0f;
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k * L + sub < cols) {
          const float dlt = v[k] - mu;
          qs = fmaf(dlt, dlt, qs);
        }
      const float var = warp_allreduce<SumF32, L>(qs) * (1.0f / (float)cols);
      const float rs = 1.0f / sqrtf(var + eps);
      if (row < rows) {
        if constexpr (MODE == kModeLayernorm) {
          uint16_t *yr = ybf + row * (int64_t)cols;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const int i = k * L + sub;
            if (i < cols) {
              const __nv_bfloat16 h =
                  __float2bfloat16_rn(fmaf((v[k] - mu) * rs, __ldg(gamma + i), __ldg(beta + i)));
              yr[i] = *reinterpret_cast<const uint16_t *>(&h);
            }
          }
        }
        if (sub == 0) {
          if (mean) mean[row] = mu;
          if (rstd) rstd[row] = rs;
        }
      }
    }
  }
}

// Chunked form, for the same rows when they span a few 16-byte chunks: a
// row is split into its head (the elements before its first 16-byte
// boundary, fewer than EPV), its whole aligned 16-byte chunks, and its tail
// (the elements after the last whole chunk).  The whole chunks are spread
// over the segment as the vectors of the vector form (lane `sub` holds
// chunks k * L + sub) and come by 16-byte loads; lane `sub` holds head and
// tail elements i * L + sub by element loads.  Every fold takes the chunks
// in order, then the head, then the tail elements, each slot under a
// predicate.  Whole chunks of the outputs go as vectors when the output
// shares x's offset within a chunk (vst: 2 for 32-byte, 1 for 16-byte
// stores), the rest element by element.  The rewrite reads gamma and beta
// from a copy each CTA makes in shared memory (their offset within a chunk
// follows the row's) and computes two elements per packed fp32 instruction.
// Shared-memory image of gamma and beta for the chunked rewrite: for each
// column pair (j, j + 1) the float4 (gamma[j], gamma[j + 1], beta[j],
// beta[j + 1]), so that one 16-byte load gives a pair's packed operands.
// Pairs start at even columns in the first image and at odd ones in the
// second (a row's chunks start at its head's parity).  Pair s of an image
// sits at slot s + s / (EPV / 2): a pad slot after each chunk's worth, so
// that lanes reading the same pair of consecutive chunks hit distinct banks.
// Whole chunk t of a row whose chunks start at pair o (o < EPV / 2) of its
// image takes its pair i from slot (EPV / 2 + 1) t + o + i + (o + i) / (EPV / 2).
__host__ __device__ constexpr int gq_slots(int cols, int epv) {
  return cols / 2 + (cols / 2) / (epv / 2) + 1;
}

template <class In, int MODE, int L, int NV>
__global__ void __launch_bounds__(kWarpRowMaxThreads)
k_rowwise_warp_ck(const typename In::S *__restrict__ x, int64_t rows, int cols, float eps,
                  float *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd,
                  const float *__restrict__ gamma, const float *__restrict__ beta,
                  uint16_t *__restrict__ ybf, int hx, int vst) {
  pdl_begin();
  using S = typename In::S;
  constexpr int EPV = In::EPV, RPW = 32 / L, HS = (EPV - 1 + L - 1) / L;
  const int lane = threadIdx.x & 31, seg = lane / L, sub = lane % L;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = (((int64_t)gridDim.x * blockDim.x) >> 5) * RPW;
  constexpr int PG = EPV / 2;      // column pairs a whole chunk
  extern __shared__ float4 sgq[];  // rewrite: the two pair images, padded
  const int gqs = gq_slots(cols, EPV);
  if constexpr (MODE == kModeLayernorm) {
    for (int par = 0; par < 2; ++par) {
      const int np = (cols - par) / 2;
      for (int q = threadIdx.x; q < np; q += blockDim.x) {
        const int j = 2 * q + par;
        sgq[par * gqs + q + q / PG] =
            make_float4(__ldg(gamma + j), __ldg(gamma + j + 1), __ldg(beta + j), __ldg(beta + j + 1));
      }
    }
    __syncthreads();
  }
  // head length of row r: the elements before its first 16-byte boundary
  auto head_of = [&](int64_t r) {
    const int lo = (int)((hx + r * (int64_t)cols) % EPV);
    const int hh = lo ? EPV - lo : 0;
    return hh < cols ? hh : cols;
  };
  uint4 raw[NV];
  S rh[HS], rt[HS];
  auto fetch = [&](int64_t r) {
    const int64_t rc = r < rows ? r : rows - 1;
    const S *xr = x + rc * (int64_t)cols;
    const int hh = head_of(rc), nw = (cols - hh) / EPV, te = hh + nw * EPV;
    const uint4 *wc = reinterpret_cast<const uint4 *>(xr + hh);
#pragma unroll
    for (int k = 0; k < NV; ++k)
      raw[k] = (k * L + sub < nw) ? ld_stream_u4(wc + k * L + sub) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < HS; ++i) {
      const int e = i * L + sub;
      rh[i] = e < hh ? __ldg(xr + e) : S(0);
      rt[i] = te + e < cols ? __ldg(xr + te + e) : S(0);
    }
  };
  int64_t r0 = warp * RPW;
  if (r0 < rows) fetch(r0 + seg);
  for (; r0 < rows; r0 += stride) {  // warp-uniform trip count
    const int64_t row = r0 + seg;
    const int hh = head_of(row < rows ? row : rows - 1), nw = (cols - hh) / EPV;
    const int te = hh + nw * EPV;
    float v[NV][EPV], h[HS], t[HS];
#pragma unroll
    for (int k = 0; k < NV; ++k) In::unpack(raw[k], v[k]);
#pragma unroll
    for (int i = 0; i < HS; ++i) { h[i] = In::cvt(rh[i]); t[i] = In::cvt(rt[i]); }
    if (r0 + stride < rows) fetch(r0 + stride + seg);
    auto whole = [&](int k) { return k * L + sub < nw; };
    auto in_head = [&](int i) { return i * L + sub < hh; };
    auto in_tail = [&](int i) { return te + i * L + sub < cols; };
    if constexpr (MODE == kModeSoftmax) {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (whole(k)) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) m = fmaxf(m, v[k][e]);
        }
#pragma unroll
      for (int i = 0; i < HS; ++i) {
        if (in_head(i)) m = fmaxf(m, h[i]);
        if (in_tail(i)) m = fmaxf(m, t[i]);
      }
      float s = 0.0f;
      if (m != -INFINITY) {
        const float mb = m * kLog2e;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          float sk = 0.0f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) {
            const float p = ex2_approx(fmaf(v[k][e], kLog2e, -mb));
            v[k][e] = p;
            sk += p;
          }
          if (whole(k)) s += sk;
        }
#pragma unroll
        for (int i = 0; i < HS; ++i) {
          h[i] = ex2_approx(fmaf(h[i], kLog2e, -mb));
          t[i] = ex2_approx(fmaf(t[i], kLog2e, -mb));
          if (in_head(i)) s += h[i];
        }
#pragma unroll
        for (int i = 0; i < HS; ++i)
          if (in_tail(i)) s += t[i];
      } else {
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
          for (int e = 0; e < EPV; ++e) v[k][e] = 0.0f;
#pragma unroll
        for (int i = 0; i < HS; ++i) h[i] = t[i] = 0.0f;
      }
      float M = m, S_ = s;
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1)
        ms_combine(M, S_, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S_, o));
      const float f = (m == -INFINITY) ? 0.0f : ex2_approx((m - M) * kLog2e) * (1.0f / S_);
      if (row < rows) {
        float *yr = y + row * (int64_t)cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          if (!whole(k)) continue;
          float *p = yr + hh + (k * L + sub) * EPV;
          float o[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) o[e] = v[k][e] * f;
          if constexpr (EPV == 8) {
            if (vst == 2) {
              st_stream_v8(p, o);
              continue;
            }
          }
          if (vst) {
#pragma unroll
            for (int e = 0; e < EPV; e += 4) st_stream_v4(p + e, o[e], o[e + 1], o[e + 2], o[e + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) p[e] = o[e];
          }
        }
#pragma unroll
        for (int i = 0; i < HS; ++i) {
          if (in_head(i)) yr[i * L + sub] = h[i] * f;
          if (in_tail(i)) yr[te + i * L + sub] = t[i] * f;
        }
      }
    } else {
      // the whole chunks two elements per packed fp32 instruction (even and
      // odd elements in the two halves), the head and tail one by one
      uint64_t sa = 0;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (whole(k)) {
#pragma unroll
          for (int i = 0; i < EPV / 2; ++i) sa = f2_add(sa, f2_pack(v[k][2 * i], v[k][2 * i + 1]));
        }
      float slo, shi;
      f2_unpack(sa, slo, shi);
      float s = slo + shi;
#pragma unroll
      for (int i = 0; i < HS; ++i)
        if (in_head(i)) s += h[i];
#pragma unroll
      for (int i = 0; i < HS; ++i)
        if (in_tail(i)) s += t[i];
      const float mu = warp_allreduce<SumF32, L>(s) / (float)cols;
      const uint64_t nmu2 = f2_pack(-mu, -mu);
      uint64_t qa = 0;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (whole(k)) {
#pragma unroll
          for (int i = 0; i < EPV / 2; ++i) {
            const uint64_t d = f2_add(f2_pack(v[k][2 * i], v[k][2 * i + 1]), nmu2);
            qa = f2_fma(d, d, qa);
          }
        }
      float qlo, qhi;
      f2_unpack(qa, qlo, qhi);
      float qs = qlo + qhi;
#pragma unroll
      for (int i = 0; i < HS; ++i)
        if (in_head(i)) {
          const float dlt = h[i] - mu;
          qs = fmaf(dlt, dlt, qs);
        }
#pragma unroll
      for (int i = 0; i < HS; ++i)
        if (in_tail(i)) {
          const float dlt = t[i] - mu;
          qs = fmaf(dlt, dlt, qs);
        }
      const float var = warp_allreduce<SumF32, L>(qs) * (1.0f / (float)cols);
      const float rs = 1.0f / sqrtf(var + eps);
      if (row < rows) {
        if constexpr (MODE == kModeLayernorm) {
          uint16_t *yr = ybf + row * (int64_t)cols;
          // the row's chunks start at column hh: pair image hh & 1, first
          // pair o = hh / 2 of it; dq[i]: slot of pair i past the chunk's base
          const float4 *img = sgq + (hh & 1) * gqs;
          const int o = hh >> 1;
          int dq[PG];
#pragma unroll
          for (int i = 0; i < PG; ++i) dq[i] = o + i + (o + i) / PG;
          const uint64_t mu2 = f2_pack(mu, mu), rs2 = f2_pack(rs, rs);
#pragma unroll
          for (int k = 0; k < NV; ++k) {
            if (!whole(k)) continue;
            const int j0 = hh + (k * L + sub) * EPV;
            const float4 *q = img + (PG + 1) * (k * L + sub);
            uint32_t pk[EPV / 2];
#pragma unroll
            for (int i = 0; i < PG; ++i) {
              // fmaf((x - mu) * rs, gamma, beta), two elements at a time
              const float4 gb = q[dq[i]];
              float lo, hi;
              f2_unpack(f2_fma(f2_mul(f2_sub(f2_pack(v[k][2 * i], v[k][2 * i + 1]), mu2), rs2),
                               f2_pack(gb.x, gb.y), f2_pack(gb.z, gb.w)), lo, hi);
              pk[i] = bf16x2_bits(lo, hi);
            }
            if (vst) {
              if constexpr (EPV == 8) {
                *reinterpret_cast<uint4 *>(yr + j0) =
                    make_uint4(pk[0], pk[1 % (EPV / 2)], pk[2 % (EPV / 2)], pk[3 % (EPV / 2)]);
              } else {
                *reinterpret_cast<uint2 *>(yr + j0) = make_uint2(pk[0], pk[1 % (EPV / 2)]);
              }
            } else {
#pragma unroll
              for (int e = 0; e < EPV; e += 2) {
                yr[j0 + e] = (uint16_t)(pk[e / 2] & 0xffffu);
                yr[j0 + e + 1] = (uint16_t)(pk[e / 2] >> 16);
              }
            }
          }
          auto put = [&](int j, float xv) {
            const __nv_bfloat16 ob =
                __float2bfloat16_rn(fmaf((xv - mu) * rs, __ldg(gamma + j), __ldg(beta + j)));
            yr[j] = *reinterpret_cast<const uint16_t *>(&ob);
          };
#pragma unroll
          for (int i = 0; i < HS; ++i) {
            if (in_head(i)) put(i * L + sub, h[i]);
            if (in_tail(i)) put(te + i * L + sub, t[i]);
          }
        }
        if (sub == 0) {
          if (mean) mean[row] = mu;
          if (rstd) rstd[row] = rs;
        }
      }
    }
  }
}

// CTAs of up to 8 warps, persistent over the rows.  With fewer rows than
// 8 warps per SM take, the CTAs shrink (down to one warp) so that the warps
// spread over every SM instead of filling a few.
template <class K>
void warp_row_launch(K k, int rpw, int64_t rows, const DevInfo &d, int *grid_out,
                     int *threads_out, size_t smem = 0) {
  const int64_t warps = (rows + rpw - 1) / rpw;
  int wpb = kWarpRowMaxThreads / 32;
  if (warps < (int64_t)wpb * d.sm_count) {
    const int64_t w = warps / d.sm_count;
    wpb = w < 1 ? 1 : (int)w;
  }
  const int threads = wpb * 32;
  const int nb = occupancy_blocks((const void *)k, threads, smem, d.device);
  const int64_t need = (warps + wpb - 1) / wpb;
  const int64_t cap = (int64_t)(nb > 0 ? nb : 1) * d.sm_count;
  *grid_out = (int)(need < cap ? need : cap);
  *threads_out = threads;
}

template <class In, int MODE, int L, int NV>
int launch_ck(const void *x, int64_t rows, int64_t cols, float eps, float *y, float *mean,
              float *rstd, const float *gamma, const float *beta, uint16_t *ybf, cudaStream_t s,
              const DevInfo &d) {
  auto k = k_rowwise_warp_ck<In, MODE, L, NV>;
  constexpr int EPV = In::EPV;
  const int hx = (int)(((uintptr_t)x / sizeof(typename In::S)) % EPV);
  // the output shares x's offset within a chunk: whole chunks store as
  // vectors (softmax of bf16: 32-byte stores when y is 32-byte aligned there)
  int vst = 0;
  if (MODE == kModeSoftmax) {
    const uintptr_t yo = ((uintptr_t)y / 4 + 8 - (uintptr_t)hx) % 8;
    vst = (EPV == 8 && yo == 0) ? 2 : (yo % 4 == 0 ? 1 : 0);
  } else if (MODE == kModeLayernorm) {
    vst = (((uintptr_t)ybf / 2) % EPV) == (uintptr_t)hx;
  }
  const size_t smem = MODE == kModeLayernorm ? 2 * sizeof(float4) * gq_slots((int)cols, EPV) : 0;
  int grid, threads;
  warp_row_launch(k, 32 / L, rows, d, &grid, &threads, smem);
  return cuda_status(launch_kernel(k, dim3(grid), dim3(threads), smem, s, 0,
                                   (const typename In::S *)x, rows, (int)cols, eps, y, mean,
                                   rstd, gamma, beta, ybf, hx, vst));
}

template <class In, int MODE, int L, int NV, bool EL = false>
int launch_one(const void *x, int64_t rows, int64_t cols, float eps, float *y, float *mean,
               float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
               cudaStream_t s, const DevInfo &d) {
  auto k = [] {
    if constexpr (EL) return k_rowwise_warp_el<In, MODE, L, NV>;
    else return k_rowwise_warp<In, MODE, L, NV>;
  }();
  int grid, threads;
  warp_row_launch(k, 32 / L, rows, d, &grid, &threads);
  return cuda_status(launch_kernel(k, dim3(grid), dim3(threads), 0, s, 0,
                                   (const typename In::S *)x, rows, (int)cols, eps, y, mean,
                                   rstd, gamma, beta, ybf));
}

template <class In, int MODE, int L>
int launch_nv(int nv, const void *x, int64_t rows, int64_t cols, float eps, float *y,
              float *mean, float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
              cudaStream_t s, const DevInfo &d) {
  switch (nv) {
    case 1: return launch_one<In, MODE, L, 1>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 2: return launch_one<In, MODE, L, 2>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 4: return launch_one<In, MODE, L, 4>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_one<In, MODE, L, 8>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

template <class In, int MODE>
int launch_mode(int L, int nv, const void *x, int64_t rows, int64_t cols, float eps, float *y,
                float *mean, float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
                cudaStream_t s, const DevInfo &d) {
  switch (L) {
    case 1: return launch_nv<In, MODE, 1>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 2: return launch_nv<In, MODE, 2>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 4: return launch_nv<In, MODE, 4>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 8: return launch_nv<In, MODE, 8>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 16: return launch_nv<In, MODE, 16>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_nv<In, MODE, 32>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

// Element-wise form: (L, K) pairs with K >= 2, 32 * 32 elements at most.
template <class In, int MODE>
int launch_mode_el(int L, int K, const void *x, int64_t rows, int64_t cols, float eps, float *y,
                   float *mean, float *rstd, const float *gamma, const float *beta,
                   uint16_t *ybf, cudaStream_t s, const DevInfo &d) {
#define RR_EL(LL, KK) \
  return launch_one<In, MODE, LL, KK, true>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d)
  if (L < 32) {
    switch (L) {
      case 1: RR_EL(1, 4);
      case 2: RR_EL(2, 4);
      case 4: RR_EL(4, 4);
      case 8: RR_EL(8, 4);
      default: RR_EL(16, 4);
    }
  }
  switch (K) {
    case 4: RR_EL(32, 4);
    case 8: RR_EL(32, 8);
    case 16: RR_EL(32, 16);
    default: RR_EL(32, 32);
  }
#undef RR_EL
}

template <class In, int MODE, int L>
int launch_ck_nv(int nv, const void *x, int64_t rows, int64_t cols, float eps, float *y,
                 float *mean, float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
                 cudaStream_t s, const DevInfo &d) {
  switch (nv) {
    case 1: return launch_ck<In, MODE, L, 1>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 2: return launch_ck<In, MODE, L, 2>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 4: return launch_ck<In, MODE, L, 4>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_ck<In, MODE, L, 8>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

template <class In, int MODE>
int launch_mode_ck(int L, int nv, const void *x, int64_t rows, int64_t cols, float eps, float *y,
                   float *mean, float *rstd, const float *gamma, const float *beta, uint16_t *ybf,
                   cudaStream_t s, const DevInfo &d) {
  switch (L) {
    case 1: return launch_ck_nv<In, MODE, 1>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 2: return launch_ck_nv<In, MODE, 2>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 4: return launch_ck_nv<In, MODE, 4>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 8: return launch_ck_nv<In, MODE, 8>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case 16: return launch_ck_nv<In, MODE, 16>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_ck_nv<In, MODE, 32>(nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

// the most whole 16-byte chunks a row holds (at least 1)
inline int64_t chunks_max(int64_t cols, int in_dtype) {
  const int64_t c = cols / (in_dtype == RR_BF16 ? 8 : 4);
  return c > 0 ? c : 1;
}

}  // namespace

int rowwise_warp_lanes(int64_t nvec, int lanes, bool rewrite) {
  if (nvec < 1 || nvec > (int64_t)32 * kRowWarpMaxNV) return 0;
  if (lanes != 0) {
    if (!(lanes == 1 || lanes == 2 || lanes == 4 || lanes == 8 || lanes == 16 || lanes == 32))
      return 0;
    return (int64_t)lanes * kRowWarpMaxNV >= nvec ? lanes : 0;
  }
  // rows of up to 8 vectors: about 2 vectors per lane; longer rows: about
  // kRowWarpTargetNV per lane, up to 32 lanes.  The layernorm rewrite, which
  // also holds gamma and beta for its vectors, takes 2 per lane throughout:
  // at 4 it needs ~120 registers and half the resident warps.
  const int per = (nvec <= 8 || rewrite) ? 2 : kRowWarpTargetNV;
  int L = 1;
  while (L < 32 && (int64_t)L * per < nvec) L *= 2;
  return L;
}

int rowwise_warp_nv(int64_t nvec, int lanes) {
  const int64_t per = (nvec + lanes - 1) / lanes;
  int nv = 1;
  while (nv < per) nv *= 2;
  return nv;
}

int rowwise_warp_el_lanes(int64_t cols, int lanes) {
  if (cols < 1 || cols > (int64_t)32 * kRowWarpMaxElPerLane) return 0;
  // 4 elements per lane up to 64 elements, then 32 lanes with 4..32 each
  int L = 1;
  while (L < 32 && (int64_t)L * 4 < cols) L *= 2;
  if (lanes == 0) return L;
  if (!(lanes == 1 || lanes == 2 || lanes == 4 || lanes == 8 || lanes == 16 || lanes == 32)) return 0;
  if (lanes < 32) return (int64_t)lanes * 4 >= cols ? lanes : 0;
  return lanes;
}

// Rows that are not aligned vectors take the chunked form while their
// chunks fit 32 lanes x 8 and the output (if any) shares x's offset within
// a chunk, the layernorm rewrite from RR_WARP_CHUNK_MIN_COLS_LN columns on;
// the element-wise form otherwise.
#ifndef RR_WARP_CHUNK_MIN_COLS_LN
#define RR_WARP_CHUNK_MIN_COLS_LN 32
#endif
static bool warp_mis_chunked(int64_t cols, int in_dtype, int mode, bool out_vec) {
  if (chunks_max(cols, in_dtype) > (int64_t)32 * kRowWarpMaxNV) return false;
  if (mode == kModeStats) return true;
  return out_vec && (mode == kModeSoftmax || cols >= RR_WARP_CHUNK_MIN_COLS_LN);
}

bool rowwise_warp_out_vec(int mode, int in_dtype, const void *x, const void *out) {
  const uintptr_t elt = in_dtype == RR_BF16 ? 2 : 4, epv = 16 / elt;
  const uintptr_t hx = ((uintptr_t)x / elt) % epv;
  if (mode == kModeSoftmax) return ((uintptr_t)out / 4 + 8 - hx) % 4 == 0;
  if (mode == kModeLayernorm) return ((uintptr_t)out / 2) % epv == hx;
  return true;
}

int rowwise_warp_mis_lanes(int64_t cols, int in_dtype, int mode, bool out_vec, int lanes) {
  if (cols < 1) return 0;
  if (warp_mis_chunked(cols, in_dtype, mode, out_vec))
    return rowwise_warp_lanes(chunks_max(cols, in_dtype), lanes, mode == kModeLayernorm);
  return rowwise_warp_el_lanes(cols, lanes);
}

int launch_rowwise_warp_mis(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                            float eps, float *y, float *mean, float *rstd, const float *gamma,
                            const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                            const DevInfo &d) {
  const bool ov = rowwise_warp_out_vec(mode, in_dtype, x, mode == kModeSoftmax ? (const void *)y
                                                                               : (const void *)ybf);
  if (!warp_mis_chunked(cols, in_dtype, mode, ov))
    return launch_rowwise_warp_el(mode, in_dtype, x, rows, cols, eps, y, mean, rstd, gamma, beta,
                                  ybf, lanes, s, d);
  const int nv = rowwise_warp_nv(chunks_max(cols, in_dtype), lanes);
  if (log_enabled())
    std::fprintf(stderr, "rr: %s warp (chunked) rows=%lld cols=%lld L=%d NV=%d\n",
                 mode == kModeSoftmax ? "softmax" : (mode == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, lanes, nv);
  if (in_dtype == RR_BF16) {
    switch (mode) {
      case kModeSoftmax: return launch_mode_ck<InBF16, kModeSoftmax>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      case kModeStats: return launch_mode_ck<InBF16, kModeStats>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      default: return launch_mode_ck<InBF16, kModeLayernorm>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    }
  }
  switch (mode) {
    case kModeSoftmax: return launch_mode_ck<InF32, kModeSoftmax>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case kModeStats: return launch_mode_ck<InF32, kModeStats>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_mode_ck<InF32, kModeLayernorm>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

int launch_rowwise_warp_el(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                           float eps, float *y, float *mean, float *rstd, const float *gamma,
                           const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                           const DevInfo &d) {
  if (cols > (int64_t)32 * kRowWarpMaxElPerLane) return RR_ERR_INVALID;
  int K = 4;
  if (lanes == 32)
    while ((int64_t)32 * K < cols) K *= 2;
  if (log_enabled())
    std::fprintf(stderr, "rr: %s warp (element-wise) rows=%lld cols=%lld L=%d K=%d\n",
                 mode == kModeSoftmax ? "softmax" : (mode == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, lanes, K);
  if (in_dtype == RR_BF16) {
    switch (mode) {
      case kModeSoftmax: return launch_mode_el<InBF16, kModeSoftmax>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      case kModeStats: return launch_mode_el<InBF16, kModeStats>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      default: return launch_mode_el<InBF16, kModeLayernorm>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    }
  }
  switch (mode) {
    case kModeSoftmax: return launch_mode_el<InF32, kModeSoftmax>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case kModeStats: return launch_mode_el<InF32, kModeStats>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_mode_el<InF32, kModeLayernorm>(lanes, K, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

int launch_rowwise_warp(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                        float eps, float *y, float *mean, float *rstd, const float *gamma,
                        const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                        const DevInfo &d) {
  const int epv = in_dtype == RR_BF16 ? 8 : 4;
  const int64_t nvec = cols / epv;
  const int nv = rowwise_warp_nv(nvec, lanes);
  if (nv > kRowWarpMaxNV || cols > 0x7fffffffLL) return RR_ERR_INVALID;
  if (log_enabled())
    std::fprintf(stderr, "rr: %s warp rows=%lld cols=%lld L=%d NV=%d\n",
                 mode == kModeSoftmax ? "softmax" : (mode == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, lanes, nv);
  if (in_dtype == RR_BF16) {
    switch (mode) {
      case kModeSoftmax: return launch_mode<InBF16, kModeSoftmax>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      case kModeStats: return launch_mode<InBF16, kModeStats>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
      default: return launch_mode<InBF16, kModeLayernorm>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    }
  }
  switch (mode) {
    case kModeSoftmax: return launch_mode<InF32, kModeSoftmax>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    case kModeStats: return launch_mode<InF32, kModeStats>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
    default: return launch_mode<InF32, kModeLayernorm>(lanes, nv, x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, s, d);
  }
}

}  // namespace rr
