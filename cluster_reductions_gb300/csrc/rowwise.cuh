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

__device__ __forceinline__ uint2 ld_stream_u2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Input element types: bf16 (held as its raw 16 bits) or fp32, read as
// 16-byte vectors (W = uint4) -- or, for rows whose base is only 8-byte
// aligned (InBF16h, InF32h), as 8-byte vectors (W = uint2).
struct InBF16 {
  using S = unsigned short;
  using W = uint4;
  static __device__ __forceinline__ W ldv(const W *p) { return ld_stream_u4(p); }
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
  static __device__ __forceinline__ float cvt(S r) { return __uint_as_float(((uint32_t)r) << 16); }
};
struct InF32 {
  using S = float;
  using W = uint4;
  static __device__ __forceinline__ W ldv(const W *p) { return ld_stream_u4(p); }
  static constexpr int EPV = 4;
  static __device__ __forceinline__ void unpack(const uint4 &w, float (&o)[4]) {
    o[0] = __uint_as_float(w.x); o[1] = __uint_as_float(w.y);
    o[2] = __uint_as_float(w.z); o[3] = __uint_as_float(w.w);
  }
  static __device__ __forceinline__ float load1(const S *p) { return __ldg(p); }
  static __device__ __forceinline__ float cvt(S r) { return r; }
};
struct InBF16h {
  using S = unsigned short;
  using W = uint2;
  static __device__ __forceinline__ W ldv(const W *p) { return ld_stream_u2(p); }
  static constexpr int EPV = 4;  // elements per 8-byte vector
  static __device__ __forceinline__ void unpack(const uint2 &w, float (&o)[4]) {
    o[0] = __uint_as_float(w.x << 16);
    o[1] = __uint_as_float(w.x & 0xffff0000u);
    o[2] = __uint_as_float(w.y << 16);
    o[3] = __uint_as_float(w.y & 0xffff0000u);
  }
  static __device__ __forceinline__ float load1(const S *p) {
    return __uint_as_float(((uint32_t)__ldg(p)) << 16);
  }
  static __device__ __forceinline__ float cvt(S r) { return __uint_as_float(((uint32_t)r) << 16); }
};
struct InF32h {
  using S = float;
  using W = uint2;
  static __device__ __forceinline__ W ldv(const W *p) { return ld_stream_u2(p); }
  static constexpr int EPV = 2;
  static __device__ __forceinline__ void unpack(const uint2 &w, float (&o)[2]) {
    o[0] = __uint_as_float(w.x);
    o[1] = __uint_as_float(w.y);
  }
  static __device__ __forceinline__ float load1(const S *p) { return __ldg(p); }
  static __device__ __forceinline__ float cvt(S r) { return r; }
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

// Xor butterfly of (max, sum) states over segments of SEG lanes;
// ms_combine is symmetric, so both lanes of a pair get the same bits.
template <int SEG>
__device__ __forceinline__ void ms_warp(float &m, float &s) {
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_combine(m, s, m2, s2);
  }
}

// ---------------------------------------------------------------------------
// Two fp32 values in one 64-bit register (the lower element in the low
// half) for the packed FP32 instructions of sm_100 and later
// ({add,sub,mul,fma}.rn.f32x2): two IEEE round-to-nearest operations per
// instruction, so every element gets exactly the bits of the scalar
// operation.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// A 32-bit word of two bf16 (the lower element in the low 16 bits) as a
// pair of fp32.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// ---------------------------------------------------------------------------
// The layernorm statistics as a monoid: (count, mean, M2), M2 the sum of
// squared deviations from the mean, merged with the update of Chan, Golub
// and LeVeque ("Updating formulae and a pairwise algorithm for computing
// sample variances", 1979): n = na + nb, d = mean_b - mean_a,
// mean = mean_a + d nb / n, M2 = M2a + M2b + d^2 na nb / n.
// ---------------------------------------------------------------------------
// Monoid state of the layernorm statistics: count, mean and M2.
struct Chan {
  uint32_t n;
  float mean, m2;
};

__device__ __forceinline__ Chan chan_merge(const Chan &a, const Chan &b) {
  if (b.n == 0) return a;
  if (a.n == 0) return b;
  Chan r;
  r.n = a.n + b.n;
  // the weight nb / n to about 2 ulp (a reciprocal and a product): its error
  // moves the mean by ~2^-23 |d|, far inside the statistics' tolerance
  const float wb = __fdividef((float)b.n, (float)r.n);
  const float d = b.mean - a.mean;
  r.mean = fmaf(d, wb, a.mean);
  r.m2 = (a.m2 + b.m2) + (d * d) * ((float)a.n * wb);
  return r;
}

// Xor butterfly over a warp's lanes (SEG a power of two); the lower lane of
// each pair is always the left operand, so both lanes of a pair compute the
// same expression and lane 0's result depends only on the lanes' values.
template <int SEG>
__device__ __forceinline__ Chan chan_warp(Chan v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) {
    Chan q;
    q.n = __shfl_xor_sync(0xffffffffu, v.n, o);
    q.mean = __shfl_xor_sync(0xffffffffu, v.mean, o);
    q.m2 = __shfl_xor_sync(0xffffffffu, v.m2, o);
    v = (lane & o) ? chan_merge(q, v) : chan_merge(v, q);
  }
  return v;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}


enum { kModeSoftmax = 0, kModeStats = 1, kModeLayernorm = 2 };

// gamma[off .. off+N) and beta[off .. off+N) of the layernorm rewrite
// (N = 2 with 8-byte, N = 4 or 8 with 16-byte aligned offsets), through the read-only path and kept in L1:
// every row reads the same values.  With both 32-byte aligned (`a32`) an
// 8-value group is one 256-bit load per array.  Lanes of a warp hold
// adjacent groups, so a warp's load spans 32 groups either way; two 128-bit
// loads per array each cover every other 16 bytes of that span and cost the
// L1 as many wavefronts as one 256-bit load, which halves the rewrite's L1
// traffic (the L1, not DRAM, bounded it).
template <int N>
__device__ __forceinline__ void load_gamma_beta(const float *__restrict__ gamma,
                                                const float *__restrict__ beta, int64_t off,
                                                bool a32, float (&g)[N], float (&b)[N]) {
  if constexpr (N == 8) {
    if (a32) {
      asm("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
          : "=f"(g[0]), "=f"(g[1]), "=f"(g[2]), "=f"(g[3]), "=f"(g[4]), "=f"(g[5]), "=f"(g[6]),
            "=f"(g[7])
          : "l"(gamma + off));
      asm("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
          : "=f"(b[0]), "=f"(b[1]), "=f"(b[2]), "=f"(b[3]), "=f"(b[4]), "=f"(b[5]), "=f"(b[6]),
            "=f"(b[7])
          : "l"(beta + off));
      return;
    }
  }
  if constexpr (N == 2) {
    const float2 gv = __ldg(reinterpret_cast<const float2 *>(gamma + off));
    const float2 bv = __ldg(reinterpret_cast<const float2 *>(beta + off));
    g[0] = gv.x; g[1] = gv.y;
    b[0] = bv.x; b[1] = bv.y;
    return;
  }
#pragma unroll
  for (int e = 0; e < N; e += 4) {
    const float4 gv = __ldg(reinterpret_cast<const float4 *>(gamma + off + e));
    const float4 bv = __ldg(reinterpret_cast<const float4 *>(beta + off + e));
    g[e] = gv.x; g[e + 1] = gv.y; g[e + 2] = gv.z; g[e + 3] = gv.w;
    b[e] = bv.x; b[e + 1] = bv.y; b[e + 2] = bv.z; b[e + 3] = bv.w;
  }
}

__device__ __forceinline__ bool aligned32(const float *a, const float *b) {
  return (((uintptr_t)a | (uintptr_t)b) & 31) == 0;
}

}  // namespace
}  // namespace rr
