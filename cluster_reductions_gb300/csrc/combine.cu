// combine.cu -- split-K attention-output combine (the
// "fa4_splitk_reduce_scatter_write" page, sm100 softmax_warp): P partial
// outputs O_p with per-row statistics (m_p, l_p) are merged as
//     out = sum_p w_p O_p / sum_p w_p l_p,  w_p = 2^((m_p - max_q m_q) * scale_log2e)
// and stored as bf16.
//
// GB300 form: a cluster of P CTAs per tile of TR rows.  CTA p stages its own
// partial tile O_p[tile, :] and its (m_p, l_p) into its own shared memory
// (one 1-D bulk copy when the tile is 16-byte granular: the local analogue of
// the page's TMEM -> shared staging), then publishes it to the cluster with
// a cluster barrier (the page's phase-0 publish, which every partition joins
// even when its band is empty).  Each CTA then owns the column band
// [p*D/P, (p+1)*D/P): it folds the P partials of that band in rank order
// 0..P-1, reading the peers' tiles through distributed shared memory, scales
// by 1/L and stores bf16.  A terminal cluster barrier keeps every CTA's tile
// alive until all peers have read it.
#include <cuda_bf16.h>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

constexpr int kCombThreads = 128;
constexpr int kTileBytes = 16384;  // staged O bytes per CTA

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(kCombThreads)
k_combine(const float *__restrict__ O, const float *__restrict__ m,
          const float *__restrict__ l, int64_t rows, int D, int TR, float scale_log2e,
          uint16_t *__restrict__ out, int use_bulk, int vec, int *err) {
  extern __shared__ __align__(128) float dyn[];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const uint32_t P = cluster_nctarank(), p = cluster_ctarank();
  const int64_t row0 = (int64_t)cluster_id_x() * TR;
  const int64_t left = rows - row0;
  const int nr = (int)(left < TR ? left : TR);
  float *sO = dyn;              // [TR][D]   own partial tile
  float *sm = sO + TR * D;      // [TR]      own m_p
  float *sl = sm + TR;          // [TR]      own l_p
  float *sw = sl + TR;          // [TR][P]   weights w_q
  float *sinv = sw + TR * P;    // [TR]      1 / L, or 0 for a dead row

  // ---- stage own partial (HBM -> own shared memory)
  const float *Op = O + ((int64_t)p * rows + row0) * D;
  bool landed = true;
  if (use_bulk) {
    if (tid == 0) {
      mbar_init(&bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)nr * (uint32_t)D * 4u;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(sO, Op, bytes, &bar);
    }
  } else {
    for (int i = tid; i < nr * D; i += kCombThreads) sO[i] = __ldg(Op + i);
  }
  for (int i = tid; i < nr; i += kCombThreads) {
    sm[i] = __ldg(m + (int64_t)p * rows + row0 + i);
    sl[i] = __ldg(l + (int64_t)p * rows + row0 + i);
  }
  if (use_bulk) {
    landed = mbar_wait_bounded(&bar, 0, kWaitBudget);
    if (!landed) set_error(err, kErrTimeout);
  }

  // ---- publish: every partition joins, band or not
  cluster_sync();

  // ---- per-row weights, in rank order, from every partition's (m, l)
  for (int i = tid; i < nr; i += kCombThreads) {
    const uint32_t am = smem_u32(sm + i), al = smem_u32(sl + i);
    float M = -INFINITY;
    for (uint32_t q = 0; q < P; ++q) M = fmaxf(M, ld_dsmem_f32(map_peer(am, q)));
    float L = 0.0f;
    for (uint32_t q = 0; q < P; ++q) {
      const float mq = ld_dsmem_f32(map_peer(am, q));
      float w;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(w) : "f"((mq - M) * scale_log2e));
      if (M == -INFINITY) w = 0.0f;
      sw[i * P + q] = w;
      L = fmaf(w, ld_dsmem_f32(map_peer(al, q)), L);
    }
    sinv[i] = (M == -INFINITY || L == 0.0f) ? 0.0f : 1.0f / L;
  }
  __syncthreads();

  // ---- own band: fold the P partials in rank order, scale, store bf16
  const int b0 = (int)((int64_t)p * D / P), b1 = (int)((int64_t)(p + 1) * D / P);
  const int bw = b1 - b0;
  if (vec) {
    const int cpr = bw >> 2;  // 4-column chunks per row
    for (int c = tid; c < nr * cpr; c += kCombThreads) {
      const int i = c / cpr, col = b0 + 4 * (c - i * cpr);
      const float *own = sO + i * D + col;
      const uint32_t a = smem_u32(own);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t q = 0; q < P; ++q) {
        const float4 v = (q == p) ? *reinterpret_cast<const float4 *>(own)
                                  : ld_dsmem_f4(map_peer(a, q));
        const float w = sw[i * P + q];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
      const float inv = sinv[i];
      uint2 pk;
      if (inv == 0.0f) {
        pk = make_uint2(0u, 0u);
      } else {
        pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      }
      *reinterpret_cast<uint2 *>(out + (row0 + i) * D + col) = pk;
    }
  } else {
    for (int c = tid; c < nr * bw; c += kCombThreads) {
      const int i = c / bw, col = b0 + (c - i * bw);
      const uint32_t a = smem_u32(sO + i * D + col);
      float acc = 0.0f;
      for (uint32_t q = 0; q < P; ++q) {
        const float v = (q == p) ? sO[i * D + col] : ld_dsmem_f32(map_peer(a, q));
        acc = fmaf(sw[i * P + q], v, acc);
      }
      const float inv = sinv[i];
      const __nv_bfloat16 h = __float2bfloat16_rn(inv == 0.0f ? 0.0f : acc * inv);
      out[(row0 + i) * D + col] = *reinterpret_cast<const uint16_t *>(&h);
    }
  }

  // ---- terminal: no CTA leaves while a peer may still read its tile
  cluster_sync();
  if (use_bulk && !landed && tid == 0) mbar_wait_bounded(&bar, 0, kWaitBudget);
}

struct CombineGeom {
  int TR;
  size_t smem;
};

CombineGeom geom(int P, int64_t rows, int D) {
  int TR = kTileBytes / (D * 4);
  if (TR < 1) TR = 1;
  if (TR > 64) TR = 64;
  if ((int64_t)TR > rows) TR = (int)rows;
  CombineGeom g;
  g.TR = TR;
  g.smem = sizeof(float) * ((size_t)TR * D + 2 * (size_t)TR + (size_t)TR * P + (size_t)TR);
  return g;
}

int prepare_kernel(int P, size_t smem) {
  cudaError_t e;
  if (P > 8) {
    e = cudaFuncSetAttribute(k_combine, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return RR_OK;
}

}  // namespace

int launch_combine(const float *O, const float *m, const float *l, int P, int64_t rows, int D,
                   float scale_log2e, uint16_t *out, cudaStream_t s, const DevInfo &d) {
  const CombineGeom g = geom(P, rows, D);
  int st = prepare_kernel(P, g.smem);
  if (st != RR_OK) return st;
  const int64_t tiles = (rows + g.TR - 1) / g.TR;
  if (tiles * P > 0x7fffffffLL) return RR_ERR_INVALID;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * P), 1, 1);
  cfg.blockDim = dim3(kCombThreads, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (P > 1) {
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_combine, &cfg);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return RR_ERR_UNSUPPORTED;
    }
    if (n < 1) return RR_ERR_UNSUPPORTED;
  }
  const int use_bulk = (D % 4 == 0) && ((uintptr_t)O % 16 == 0);
  const int vec = (D % P == 0) && ((D / P) % 4 == 0) && ((uintptr_t)out % 8 == 0);
  return cuda_status(cudaLaunchKernelEx(&cfg, k_combine, O, m, l, rows, D, g.TR, scale_log2e,
                                        out, use_bulk, vec, d.err_word));
}

}  // namespace rr
