// axis.cu -- monoid reduction over a non-last axis of a dense 3-D view
// x[outer][axis][inner] (the "reduce" page, algorithm/gpu/rowwise, Args:
// row_coords pins every dimension but ctx.axis, the reduce axis).
//
// The "rows" of this reduction are the outer * inner strided lines
// x[o, :, i]; consecutive i are adjacent in memory.  The page's tiers map
// onto that layout as follows:
//   tiled / serial  a thread owns E adjacent rows (i .. i+E-1) and walks the
//                   axis, one E-wide load per axis step, no cross-thread
//                   combine (E = emit_tile_width; E = 1 is the serial tier:
//                   one thread, one row);
//   warp            a warp owns a tile of L*V adjacent rows of one o; lane
//                   segments of L lanes take 32/L axis positions per step and
//                   combine with an xor butterfly (for inner 2, 3, 5, 6 or 7
//                   the slab form: a warp, or a CTA, owns the whole
//                   contiguous slab x[o, :, :] and reads it with 16-byte
//                   loads);
//   block           a CTA owns a tile; its 8 warps split the axis further and
//                   combine through shared memory in warp order;
//   split-K         a cluster of C CTAs owns a tile; each CTA folds one
//                   contiguous chunk of the axis as in the block tier, then
//                   every row of the tile is folded over ranks 0..C-1, in
//                   rank order, by the rank that owns it (row j of the tile
//                   belongs to rank j mod C), reading the peers' partials
//                   through distributed shared memory ("cluster_allreduce"
//                   page, with the result scattered instead of replicated).
//                   With G > 1 clusters per tile, the G cluster results go to
//                   a workspace and a second kernel folds them in order.
// Each thread folds its axis positions in chunks of kChunk consecutive ones
// and then folds the chunk results, so fp32 sums stay within a few units of
// rounding of the exact sum relative to ||x[o,:,i]||_2 even for very long
// axes.  Every fold order depends only on the shape, the tier, V, L, C and
// G, so a call gives the same bits on every run.
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

constexpr int kAxisThreads = 256, kAxisWarps = kAxisThreads / 32;
#ifndef RR_AXIS_UNROLL
#define RR_AXIS_UNROLL 8
#endif
#ifndef RR_AXIS_TILED_UNROLL
#define RR_AXIS_TILED_UNROLL 8
#endif
constexpr int kAxisUnroll = RR_AXIS_UNROLL, kTiledUnroll = RR_AXIS_TILED_UNROLL;
#ifndef RR_AXIS_CHUNK
#define RR_AXIS_CHUNK 1024
#endif
constexpr int kChunk = RR_AXIS_CHUNK;  // axis positions a thread folds before a chunk fold

template <class T, int V> struct VecOf;
template <> struct VecOf<float, 2> { using type = float2; };
template <> struct VecOf<int, 2> { using type = int2; };

// V adjacent elements from p (p aligned to V * 4 bytes).
template <class T, int V>
__device__ __forceinline__ void load_v(const T *p, T (&o)[V]) {
  if constexpr (V == 4) {
    const auto v = ld_stream(reinterpret_cast<const typename Vec4<T>::type *>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else if constexpr (V == 2) {
    const auto v = __ldg(reinterpret_cast<const typename VecOf<T, 2>::type *>(p));
    o[0] = v.x; o[1] = v.y;
  } else {
    o[0] = __ldg(p);
  }
}

// ---------------------------------------------------------------------------
// Tiled / serial tier.  Thread g owns rows (o, i .. i+E-1) with
// g = o * (inner / E) + i / E; it folds axis positions 0, 1, 2, ... in order
// (U loads in flight, folded in axis order).
// ---------------------------------------------------------------------------
template <class Op, int E>
__global__ void __launch_bounds__(kAxisThreads)
k_axis_tiled(const typename Op::T *__restrict__ x, int64_t outer, int64_t axis,
             int64_t inner, typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  const int64_t gpo = inner / E;
  const int64_t groups = outer * gpo;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
    const int64_t o = g / gpo, i = (g - o * gpo) * E;
    const T *p = x + o * axis * inner + i;
    T acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = Op::id();
    for (int64_t a = 0; a < axis;) {
      const int64_t a_end = a + kChunk < axis ? a + kChunk : axis;
      T ch[E];
#pragma unroll
      for (int e = 0; e < E; ++e) ch[e] = Op::id();
      for (; a + kTiledUnroll <= a_end; a += kTiledUnroll) {
        T v[kTiledUnroll][E];
#pragma unroll
        for (int u = 0; u < kTiledUnroll; ++u) load_v<T, E>(p + (a + u) * inner, v[u]);
#pragma unroll
        for (int u = 0; u < kTiledUnroll; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) ch[e] = Op::f(ch[e], v[u][e]);
      }
      for (; a < a_end; ++a) {
        T v[E];
        load_v<T, E>(p + a * inner, v);
#pragma unroll
        for (int e = 0; e < E; ++e) ch[e] = Op::f(ch[e], v[e]);
      }
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = Op::f(acc[e], ch[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) out[o * inner + i + e] = Op::finalize(acc[e]);
  }
}

// ---------------------------------------------------------------------------
// Warp, block and split-K tiers.  WPU = warps per unit (1: warp tier;
// kAxisWarps: block / split-K).  A unit is (o, tile t) with the tile's rows
// i in [t*TW, t*TW + TW), TW = L*V, L = 2^lg_L lanes per axis position.
// The axis of a unit is cut into G*C chunks: cluster split g, rank r folds
// chunk g*C + r.  Lane (sr, sc) = (lane / L, lane % L) owns rows
// t*TW + sc*V .. +V-1 and axis positions a0 + sr, a0 + sr + R*WPU, ... of its
// chunk (R = 32 / L).  Fold order per row: each thread in axis order (in
// chunks); xor butterfly over sr; warps 0..WPU-1 in order; ranks 0..C-1 in
// order; with G > 1 the G split results go to ws[g][o*inner + i] and
// k_axis_fold folds them in order g = 0..G-1.
// ---------------------------------------------------------------------------
// Block / split-K CTAs are held to 64 registers (4 resident per SM); the
// warp tier is left to the compiler, which keeps more loads in flight there.
#ifndef RR_AXIS_MIN_BLOCKS
#define RR_AXIS_MIN_BLOCKS 4
#endif
template <class Op, int V, int WPU>
__global__ void __launch_bounds__(kAxisThreads, WPU == 1 ? 1 : RR_AXIS_MIN_BLOCKS)
k_axis_coop(const typename Op::T *__restrict__ x, int64_t outer, int64_t axis,
            int64_t inner, int lg_L, int G, typename Op::T *__restrict__ out,
            typename Op::T *__restrict__ ws) {
  pdl_begin();
  using T = typename Op::T;
  __shared__ T part[WPU][32 * V];
  __shared__ T slot[2][32 * V];
  const int L = 1 << lg_L, R = 32 >> lg_L, TW = L * V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sc = lane & (L - 1), sr = lane >> lg_L;
  const int64_t ntiles = (inner + TW - 1) / TW;
  const int64_t units = outer * ntiles;
  uint32_t C = 1, rank = 0;
  int64_t worker, nworkers;
  int wsub = 0;
  if (WPU == 1) {
    worker = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    nworkers = ((int64_t)gridDim.x * blockDim.x) >> 5;
  } else {
    C = cluster_nctarank();
    rank = cluster_ctarank();
    worker = blockIdx.x / C;
    nworkers = gridDim.x / C;
    wsub = warp;
  }
  const int64_t K = (int64_t)G * C;
  const int64_t chunk = (axis + K - 1) / K;
  const int64_t AS = (int64_t)R * WPU, step = (int64_t)kAxisUnroll * AS;
  const int64_t items = units * G;
  int sel = 0;
  for (int64_t w = worker; w < items; w += nworkers) {
    const int64_t u = w / G, g = w - u * G;
    const int64_t o = u / ntiles, t = u - o * ntiles;
    const int64_t c = t * TW + sc * V;
    const int64_t kc = g * C + rank;
    const int64_t a_lo = kc * chunk < axis ? kc * chunk : axis;
    const int64_t a_hi = a_lo + chunk < axis ? a_lo + chunk : axis;
    T acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = Op::id();
    if (c < inner) {
      const T *p = x + o * axis * inner + c;
      int64_t a0 = a_lo + wsub * R + sr;
      while (a0 < a_hi) {
        T ch[V];
#pragma unroll
        for (int e = 0; e < V; ++e) ch[e] = Op::id();
        for (int it = 0; it < kChunk / kAxisUnroll && a0 < a_hi; ++it, a0 += step) {
          // The loads are unconditional, so they go out back to back: a
          // position past the end of the chunk re-reads the last one (a
          // valid address) and the fold skips it.
          const int64_t last = a_hi - 1;
          T v[kAxisUnroll][V];
#pragma unroll
          for (int k = 0; k < kAxisUnroll; ++k) {
            const int64_t a = a0 + k * AS < last ? a0 + k * AS : last;
            load_v<T, V>(p + a * inner, v[k]);
          }
#pragma unroll
          for (int k = 0; k < kAxisUnroll; ++k)
            if (a0 + k * AS < a_hi)
#pragma unroll
              for (int e = 0; e < V; ++e) ch[e] = Op::f(ch[e], v[k][e]);
        }
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = Op::f(acc[e], ch[e]);
      }
    }
    for (int off = L; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = Op::f(acc[e], shfl_xor(acc[e], off));
    if (WPU == 1) {
      if (sr == 0 && c < inner)
#pragma unroll
        for (int e = 0; e < V; ++e) out[o * inner + c + e] = Op::finalize(acc[e]);
      continue;
    }
    if (sr == 0)
#pragma unroll
      for (int e = 0; e < V; ++e) part[warp][sc * V + e] = acc[e];
    __syncthreads();
    const int j = threadIdx.x;
    T res = Op::id();
    if (j < TW) {
      res = part[0][j];
#pragma unroll
      for (int w = 1; w < WPU; ++w) res = Op::f(res, part[w][j]);
    }
    const int64_t col = t * TW + j;
    // G == 1: the final value; G > 1: this split's partial, folded later
    T *dst = G == 1 ? out : ws + g * outer * inner;
    if (C == 1) {
      if (j < TW && col < inner) dst[o * inner + col] = G == 1 ? Op::finalize(res) : res;
      __syncthreads();
      continue;
    }
    // Two slots alternate between consecutive units, so no trailing barrier
    // is needed per unit: a CTA that runs ahead writes the other slot, and
    // it cannot get two units ahead because the next barrier waits for every
    // peer.  The kernel ends with a cluster barrier.
    T *sl = slot[sel];
    if (j < TW) sl[j] = res;
    cluster_sync();
    if (j < TW && (uint32_t)j % C == rank) {
      const uint32_t addr = smem_u32(&sl[j]);
      uint32_t b[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if ((uint32_t)q < C) b[q] = ld_dsmem_u32(map_peer(addr, (uint32_t)q));
      T r = from_bits<T>(b[0]);
#pragma unroll
      for (int q = 1; q < 16; ++q)
        if ((uint32_t)q < C) r = Op::f(r, from_bits<T>(b[q]));
      if (col < inner) dst[o * inner + col] = G == 1 ? Op::finalize(r) : r;
    }
    sel ^= 1;
  }
  if (WPU > 1 && C > 1) cluster_sync();
}

// Second pass of G > 1: out[n] = ws[0][n] (+) ws[1][n] (+) ... (+) ws[G-1][n].
template <class Op>
__global__ void __launch_bounds__(kAxisThreads)
k_axis_fold(const typename Op::T *__restrict__ ws, int64_t n, int G,
            typename Op::T *__restrict__ out) {
  pdl_begin();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  typename Op::T acc = ws[i];
  for (int g = 1; g < G; ++g) acc = Op::f(acc, ws[(int64_t)g * n + i]);
  out[i] = Op::finalize(acc);
}

template <class Op>
int launch_axis_tiled(const void *xv, int64_t outer, int64_t axis, int64_t inner, void *outv,
                      int E, cudaStream_t s, const DevInfo &d) {
  using T = typename Op::T;
  const T *x = static_cast<const T *>(xv);
  T *out = static_cast<T *>(outv);
  const void *fn = E == 4 ? (const void *)k_axis_tiled<Op, 4>
                 : E == 2 ? (const void *)k_axis_tiled<Op, 2>
                          : (const void *)k_axis_tiled<Op, 1>;
  const int64_t groups = outer * (inner / E);
  const int occ = occupancy_blocks(fn, kAxisThreads, 0, d.device);
  int64_t grid = (groups + kAxisThreads - 1) / kAxisThreads;
  const int64_t cap = (int64_t)occ * d.sm_count;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  if (log_enabled())
    std::fprintf(stderr, "[rr] axis tiled E=%d outer=%lld axis=%lld inner=%lld grid=%lld\n", E,
                 (long long)outer, (long long)axis, (long long)inner, (long long)grid);
  if (E == 4)
    launch_kernel(k_axis_tiled<Op, 4>, dim3((unsigned)grid), dim3(kAxisThreads), 0, s, 0, x, outer, axis, inner, out);
  else if (E == 2)
    launch_kernel(k_axis_tiled<Op, 2>, dim3((unsigned)grid), dim3(kAxisThreads), 0, s, 0, x, outer, axis, inner, out);
  else
    launch_kernel(k_axis_tiled<Op, 1>, dim3((unsigned)grid), dim3(kAxisThreads), 0, s, 0, x, outer, axis, inner, out);
  return cuda_status(cudaGetLastError());
}

template <class Op, int V>
int launch_axis_coop(const void *xv, int64_t outer, int64_t axis, int64_t inner, void *outv,
                     const AxisPlan &pl, void *wsv, cudaStream_t s, const DevInfo &d) {
  using T = typename Op::T;
  const T *x = static_cast<const T *>(xv);
  T *out = static_cast<T *>(outv);
  T *ws = static_cast<T *>(wsv);
  const int lg_L = pl.lg_L, G = pl.G, C = pl.C;
  const int64_t TW = ((int64_t)1 << lg_L) * V;
  const int64_t units = outer * ((inner + TW - 1) / TW);
  const int64_t items = units * G;
  cudaError_t e = cudaSuccess;
  if (pl.tier == RR_TIER_WARP) {
    auto kern = k_axis_coop<Op, V, 1>;
    const int occ = occupancy_blocks((const void *)kern, kAxisThreads, 0, d.device);
    int64_t grid = (units + kAxisWarps - 1) / kAxisWarps;
    const int64_t cap = (int64_t)occ * d.sm_count;
    if (grid > cap) grid = cap;
    if (log_enabled())
      std::fprintf(stderr, "[rr] axis warp V=%d L=%d units=%lld grid=%lld\n", V, 1 << lg_L,
                   (long long)units, (long long)grid);
    launch_kernel(kern, dim3((unsigned)grid), dim3(kAxisThreads), 0, s, 0, x, outer, axis, inner, lg_L, 1, out, nullptr);
    return cuda_status(cudaGetLastError());
  }
  auto kern = k_axis_coop<Op, V, kAxisWarps>;
  if (C <= 1) {
    const int occ = occupancy_blocks((const void *)kern, kAxisThreads, 0, d.device);
    int64_t grid = items;
    const int64_t cap = (int64_t)occ * d.sm_count;
    if (grid > cap) grid = cap;
    if (log_enabled())
      std::fprintf(stderr, "[rr] axis block V=%d L=%d G=%d units=%lld grid=%lld\n", V,
                   1 << lg_L, G, (long long)units, (long long)grid);
    launch_kernel(kern, dim3((unsigned)grid), dim3(kAxisThreads), 0, s, 0, x, outer, axis, inner, lg_L, G, out, ws);
    e = cudaGetLastError();
  } else {
    if (C > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_status(e);
    }
    const int ncl = occupancy_clusters((const void *)kern, kAxisThreads, 0, C, d.device);
    if (ncl <= 0) return RR_ERR_UNSUPPORTED;
    const int64_t clusters = items < ncl ? items : ncl;
    if (log_enabled())
      std::fprintf(stderr, "[rr] axis split-K V=%d L=%d C=%d G=%d units=%lld clusters=%lld\n",
                   V, 1 << lg_L, C, G, (long long)units, (long long)clusters);
    e = launch_kernel(kern, dim3((unsigned)(clusters * C)), dim3(kAxisThreads), 0, s, C, x, outer,
                      axis, inner, lg_L, G, out, ws);
  }
  if (e != cudaSuccess || G == 1) return cuda_status(e);
  const int64_t n = outer * inner;
  launch_kernel(k_axis_fold<Op>, dim3((unsigned)((n + kAxisThreads - 1) / kAxisThreads)), dim3(kAxisThreads), 0, s, 0, 
      ws, n, G, out);
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Warp tier, slab form, for narrow inner widths that are not a multiple of 4
// (INNER = 2, 3, 5, 6, 7): WPS warps (1, or a CTA of 8) own the whole slab
// x[o, :, :], which is contiguous (axis * INNER elements).  Four axis
// positions are exactly INNER 16-byte vectors, so thread t of the slab's
// WPS * 32 reads groups t, t + WPS * 32, ... of 4 positions with vector
// loads (a warp instruction covers 512 contiguous bytes) and folds element
// e of a group into column e % INNER -- a fixed pattern.  The U groups a
// thread has in flight fold into U separate accumulator sets (independent
// dependency chains), joined in order u = 0..U-1 at each chunk end, then the
// chunks in order; the axis % 4 tail positions go one per thread.  Every
// column is then combined over the warp with an xor butterfly and, for
// WPS = 8, over the warps in warp order through shared memory.  Needs x
// 16-byte aligned and axis * INNER % 4 == 0 (every slab 16-byte aligned).
// ---------------------------------------------------------------------------
template <class Op, int INNER, int WPS>
__global__ void __launch_bounds__(kAxisThreads)
k_axis_slab(const typename Op::T *__restrict__ x, int64_t outer, int64_t axis,
            typename Op::T *__restrict__ out) {
  pdl_begin();
  using T = typename Op::T;
  using V = typename Vec4<T>::type;
  constexpr int U = 4;                              // groups in flight per thread
  constexpr int TPS = WPS * 32;                     // threads per slab
  constexpr int64_t kGroupChunk = (int64_t)(kChunk / 4) * (TPS / 32);  // groups per chunk
  __shared__ T red[WPS][INNER];
  const int lane = threadIdx.x & 31;
  const int t = WPS == 1 ? lane : (int)threadIdx.x;  // this thread's index within its slab
  const int64_t unit = ((int64_t)blockIdx.x * kAxisThreads + threadIdx.x) / TPS;
  const int64_t nunits = ((int64_t)gridDim.x * kAxisThreads) / TPS;
  const int64_t ng = axis >> 2;                     // whole groups of 4 positions
  for (int64_t o = unit; o < outer; o += nunits) {  // uniform over the slab's threads
    const T *slab = x + o * axis * INNER;
    const V *q = reinterpret_cast<const V *>(slab);
    T acc[INNER];
#pragma unroll
    for (int c = 0; c < INNER; ++c) acc[c] = Op::id();
    for (int64_t c0 = 0; c0 < ng; c0 += kGroupChunk) {
      const int64_t c1 = c0 + kGroupChunk < ng ? c0 + kGroupChunk : ng;
      T part[U][INNER];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int c = 0; c < INNER; ++c) part[u][c] = Op::id();
      for (int64_t g0 = c0 + t; g0 < c1; g0 += (int64_t)TPS * U) {
        V v[U][INNER];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t g = g0 + (int64_t)TPS * u;
          const int64_t gc = g < c1 ? g : c1 - 1;   // clamped: loads stay unconditional
#pragma unroll
          for (int k = 0; k < INNER; ++k) v[u][k] = ld_stream(q + gc * INNER + k);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (g0 + (int64_t)TPS * u < c1) {
#pragma unroll
            for (int k = 0; k < INNER; ++k) {
              part[u][(4 * k + 0) % INNER] = Op::f(part[u][(4 * k + 0) % INNER], v[u][k].x);
              part[u][(4 * k + 1) % INNER] = Op::f(part[u][(4 * k + 1) % INNER], v[u][k].y);
              part[u][(4 * k + 2) % INNER] = Op::f(part[u][(4 * k + 2) % INNER], v[u][k].z);
              part[u][(4 * k + 3) % INNER] = Op::f(part[u][(4 * k + 3) % INNER], v[u][k].w);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int c = 0; c < INNER; ++c) acc[c] = Op::f(acc[c], part[u][c]);
    }
    const int64_t pos = ng * 4 + t;                 // the axis % 4 tail positions
    if (pos < axis) {
#pragma unroll
      for (int c = 0; c < INNER; ++c) acc[c] = Op::f(acc[c], __ldg(slab + pos * INNER + c));
    }
#pragma unroll
    for (int c = 0; c < INNER; ++c) acc[c] = warp_allreduce<Op, 32>(acc[c]);
    if constexpr (WPS == 1) {
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < INNER; ++c) out[o * INNER + c] = Op::finalize(acc[c]);
      }
    } else {
      const int w = threadIdx.x >> 5;
      if (lane == 0) {
#pragma unroll
        for (int c = 0; c < INNER; ++c) red[w][c] = acc[c];
      }
      __syncthreads();
      if (threadIdx.x < INNER) {
        T r = red[0][threadIdx.x];
#pragma unroll
        for (int ww = 1; ww < WPS; ++ww) r = Op::f(r, red[ww][threadIdx.x]);
        out[o * INNER + threadIdx.x] = Op::finalize(r);
      }
      __syncthreads();
    }
  }
}

template <class Op, int INNER>
int launch_axis_slab_n(const void *x, int64_t outer, int64_t axis, void *out, bool cta,
                       cudaStream_t s, const DevInfo &d) {
  auto run = [&](auto k, int per_block) {
    const int nb = occupancy_blocks((const void *)k, kAxisThreads, 0, d.device);
    const int64_t need = (outer + per_block - 1) / per_block;
    const int64_t cap = (int64_t)(nb > 0 ? nb : 1) * d.sm_count;
    const int grid = (int)(need < cap ? need : cap);
    if (log_enabled())
      std::fprintf(stderr, "rr: axis slab outer=%lld axis=%lld inner=%d %s ctas=%d\n",
                   (long long)outer, (long long)axis, INNER, cta ? "cta" : "warp", grid);
    return cuda_status(launch_kernel(k, dim3(grid), dim3(kAxisThreads), 0, s, 0,
                                     (const typename Op::T *)x, outer, axis,
                                     (typename Op::T *)out));
  };
  if (cta) return run(k_axis_slab<Op, INNER, kAxisWarps>, 1);
  return run(k_axis_slab<Op, INNER, 1>, kAxisWarps);
}

template <class Op>
int launch_axis_slab(const void *x, int64_t outer, int64_t axis, int64_t inner, void *out,
                     bool cta, cudaStream_t s, const DevInfo &d) {
  switch (inner) {
    case 2: return launch_axis_slab_n<Op, 2>(x, outer, axis, out, cta, s, d);
    case 3: return launch_axis_slab_n<Op, 3>(x, outer, axis, out, cta, s, d);
    case 5: return launch_axis_slab_n<Op, 5>(x, outer, axis, out, cta, s, d);
    case 6: return launch_axis_slab_n<Op, 6>(x, outer, axis, out, cta, s, d);
    case 7: return launch_axis_slab_n<Op, 7>(x, outer, axis, out, cta, s, d);
    default: return RR_ERR_INVALID;
  }
}

template <class Op>
int launch_axis_op(const void *x, int64_t outer, int64_t axis, int64_t inner, void *out,
                   const AxisPlan &pl, void *ws, cudaStream_t s, const DevInfo &d) {
  if (pl.tier == RR_TIER_TILED)
    return launch_axis_tiled<Op>(x, outer, axis, inner, out, pl.E, s, d);
  if (pl.slab) return launch_axis_slab<Op>(x, outer, axis, inner, out, pl.tier == RR_TIER_BLOCK, s, d);
  if (pl.V == 4) return launch_axis_coop<Op, 4>(x, outer, axis, inner, out, pl, ws, s, d);
  return launch_axis_coop<Op, 1>(x, outer, axis, inner, out, pl, ws, s, d);
}

template <class Op>
int max_axis_cluster_for(int want, const DevInfo &d) {
  auto kern = k_axis_coop<Op, 4, kAxisWarps>;
  for (int C = 16; C >= 2; C >>= 1) {
    if (C > want) continue;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                     cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (occupancy_clusters((const void *)kern, kAxisThreads, 0, C, d.device) > 0) return C;
  }
  return 1;
}

}  // namespace

int axis_max_cluster(int want, const DevInfo &d) {
  if (!d.cluster_launch) return 1;
  return max_axis_cluster_for<SumF32>(want, d);
}

int launch_reduce_axis(const void *x, int64_t outer, int64_t axis, int64_t inner, int op,
                       int dtype, void *out, const AxisPlan &pl, void *ws, cudaStream_t s,
                       const DevInfo &d) {
  if (dtype == RR_F32) {
    if (op == RR_OP_SUM) return launch_axis_op<SumF32>(x, outer, axis, inner, out, pl, ws, s, d);
    if (op == RR_OP_MAX) return launch_axis_op<MaxF32>(x, outer, axis, inner, out, pl, ws, s, d);
    return launch_axis_op<MinF32>(x, outer, axis, inner, out, pl, ws, s, d);
  }
  if (op == RR_OP_SUM) return launch_axis_op<SumI32>(x, outer, axis, inner, out, pl, ws, s, d);
  if (op == RR_OP_MAX) return launch_axis_op<MaxI32>(x, outer, axis, inner, out, pl, ws, s, d);
  return launch_axis_op<MinI32>(x, outer, axis, inner, out, pl, ws, s, d);
}

}  // namespace rr
