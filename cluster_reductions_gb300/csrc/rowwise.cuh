// rowwise.cuh -- pieces shared by the block / split-K tiers (rowwise.cu)
// and the warp tier (rowwarp.cu) of the two-pass row operations of the
// "reduce" page (algorithm/gpu/rowwise): the input element types, the
// online-softmax (max, sum) monoid and the bf16 packing of the layernorm
// rewrite.
#pragma once

#include <cuda_bf16.h>

#include "rr_device.cuh"

namespace rr {
namespace {

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

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}


enum { kModeSoftmax = 0, kModeStats = 1, kModeLayernorm = 2 };

}  // namespace
}  // namespace rr
