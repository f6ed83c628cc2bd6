// combine.cu -- split-K attention-output combine (the
// "fa4_splitk_reduce_scatter_write" page, sm100 softmax_warp): P partial
// outputs O_p with per-row statistics (m_p, l_p) are merged as
//     out = sum_p w_p O_p / sum_p w_p l_p,  w_p = 2^((m_p - max_q m_q) * scale_log2e)
// and stored as bf16.
//
// GB300 form: a cluster of P CTAs works on tiles of TR rows.  For each tile,
// CTA p stages its own partial O_p[tile, :] into its own shared memory (the
// local analogue of the page's TMEM -> shared staging) and publishes it to
// the cluster (the page's phase-0 publish, which every partition joins even
// when its band is empty).  Each CTA owns the column band [p*D/P, (p+1)*D/P):
// it folds the P partials of that band in rank order 0..P-1, reading the
// peers' tiles through distributed shared memory (the reduce-scatter), scales
// by 1/L and stores bf16.  No CTA leaves while a peer may still read its
// shared memory.
//
// Fast path (P in {1,2,4,8,16}, D % 4P == 0, 16-byte aligned partials):
// persistent clusters stride over the tiles through a ring of kStages
// staging slots.  A producer warp stages tiles with 1-D bulk copies up to
// kStages ahead.  Each slot also receives the (m, l) of every partition for
// the tile rows (a few hundred bytes), so the weights are computed once per
// row from local shared memory and only the O band crosses DSMEM.  The
// publish and the "every peer is done with this slot" signals are mbarrier
// arrivals sent to each peer (as the page's publish_mbar), spread over the
// lanes of one warp, so no all-thread cluster barrier is needed per tile.
// Generic path: one tile per cluster, plain loads, scalar bands (any P <= 16,
// any D, bands of unequal width, empty bands when D < P).
// Two more variants compute the same bits: push (each CTA bulk-copies its
// peers' row slices into their shared memory) and direct, the default (no
// exchange at all: a CTA stages the tile rows of all P partitions and folds
// them locally; same DRAM bytes, no per-tile cluster synchronisation).
#include <cstdio>

#include <cuda_bf16.h>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"

namespace rr {
namespace {

constexpr int kCombThreads = 128;  // generic path
#ifndef RR_COMBINE_TILE_BYTES
#define RR_COMBINE_TILE_BYTES 16384
#endif
#ifndef RR_COMBINE_STAGES
#define RR_COMBINE_STAGES 3
#endif
#ifndef RR_COMBINE_CONSUMERS
#define RR_COMBINE_CONSUMERS 128
#endif
constexpr int kTileBytes = RR_COMBINE_TILE_BYTES;  // staged O bytes per CTA and slot
constexpr int kStages = RR_COMBINE_STAGES;         // staging slots per CTA (cluster variants)
constexpr int kCons = RR_COMBINE_CONSUMERS;        // consumer threads (the first warps)
constexpr int kPipeThreads = kCons + 64;           // + producer warp + publisher warp

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Weights of the tile rows from the staged (m, l) of all P partitions:
// sw[i*P + q] = w_q = 2^((m_q - M) * s) and sinv[i] = 1 / L with
// L = sum_q w_q l_q folded in rank order (0 for M = -inf or L = 0).
template <int P>
__device__ __forceinline__ void row_weights(const float *mall, const float *lall, int TRp, int nr,
                                            float scale_log2e, float *sw, float *sinv) {
  for (int i = threadIdx.x; i < nr; i += kCons) {
    float mq[P];
#pragma unroll
    for (int q = 0; q < P; ++q) mq[q] = mall[q * TRp + i];
    float M = mq[0];
#pragma unroll
    for (int q = 1; q < P; ++q) M = fmaxf(M, mq[q]);
    float L = 0.0f;
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const float w = (M == -INFINITY) ? 0.0f : ex2f_approx((mq[q] - M) * scale_log2e);
      sw[i * P + q] = w;
      L = fmaf(w, lall[q * TRp + i], L);
    }
    sinv[i] = (M == -INFINITY || L == 0.0f) ? 0.0f : 1.0f / L;
  }
}

// Fold of this CTA's band of one staged tile, 4-column chunks: the P band
// vectors (own from shared memory, peers' through DSMEM) are all loaded
// before the rank-order FMAs, so the P - 1 remote loads are in flight
// together.
template <int P>
__device__ __forceinline__ void fold_band(const float *so, int nr, int D, const float *sw,
                                          const float *sinv, uint32_t p,
                                          uint16_t *__restrict__ out_tile) {
  const int bw = D / P, cpr = bw >> 2, b0 = (int)p * bw;
  for (int c = threadIdx.x; c < nr * cpr; c += kCons) {
    const int i = c / cpr, col = b0 + 4 * (c - i * cpr);
    const float *own = so + i * D + col;
    const uint32_t ao = smem_u32(own);
    float4 v[P];
#pragma unroll
    for (int q = 0; q < P; ++q)
      v[q] = (q == (int)p) ? *reinterpret_cast<const float4 *>(own) : ld_dsmem_f4(map_peer(ao, q));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const float w = sw[i * P + q];
      acc.x = fmaf(w, v[q].x, acc.x);
      acc.y = fmaf(w, v[q].y, acc.y);
      acc.z = fmaf(w, v[q].z, acc.z);
      acc.w = fmaf(w, v[q].w, acc.w);
    }
    const float inv = sinv[i];
    uint2 pk = make_uint2(0u, 0u);
    if (inv != 0.0f) {
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    }
    *reinterpret_cast<uint2 *>(out_tile + (int64_t)i * D + col) = pk;
  }
}

// Persistent, pipelined fast path.  Slot s of every CTA holds one staged
// tile: O_p[tile, :] (TR x D), then m_q[tile] for q = 0..P-1, then l_q[tile]
// (each TRp floats, TRp = TR rounded up to 4).  Three mbarriers per slot:
//   full[s]  (local, tx-counted)  this CTA's bulk copies have landed;
//   pub[s]   (P arrivals)         every CTA's O tile of this round has landed
//                                 (warp 0 of each CTA arrives on every
//                                 peer's pub[s] once its full[s] completes);
//   cons[s]  (P arrivals)         every CTA has finished reading this CTA's
//                                 slot s, so it may be refilled.
// A barrier phase can never run two phases ahead of its waiter (each refill
// waits on cons, which needs every consumer), so parity waits are
// unambiguous.  Every wait is bounded; after the first timeout the CTA stops
// waiting (results are then garbage and the device error word says so).
// ml_bulk: (m, l) are copied by the bulk engine too (rows % 4 == 0 and
// 16-byte aligned m, l); otherwise the producer warp loads them and arrives
// on full[s] after them.
template <int P>
__global__ void __launch_bounds__(kPipeThreads)
k_combine_pipe(const float *__restrict__ O, const float *__restrict__ m,
               const float *__restrict__ l, int64_t rows, int D, int TR, float scale_log2e,
               uint16_t *__restrict__ out, int ml_bulk, int *err) {
  pdl_begin();
  extern __shared__ __align__(128) float dyn[];
  __shared__ __align__(8) uint64_t full[kStages], pub[kStages], cons[kStages];
  __shared__ int dead;
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t p = cluster_ctarank();
  const int64_t cl = cluster_id_x(), ncl = cluster_nid_x();
  const int64_t ntiles = (rows + TR - 1) / TR;
  const int TRp = (TR + 3) & ~3;
  const int slot_floats = TR * D + 2 * P * TRp;
  float *sw = dyn + kStages * slot_floats;  // [TR][P]
  float *sinv = sw + TR * P;                // [TR]
  if (tid == 0) {
    dead = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&pub[s], P);
      mbar_init(&cons[s], P);
    }
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every peer's barriers exist before any remote arrive

  const int64_t K = (cl < ntiles) ? (ntiles - 1 - cl) / ncl + 1 : 0;  // tiles of this cluster
  if (tid >= kCons + 32) {
    // ---- publisher warp: once this CTA's copies of a tile have landed,
    // arrive on every peer's pub[s] (one lane per peer).  It issues no
    // global stores, so its cluster-scope release has nothing to wait for.
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t par = (uint32_t)(k / kStages) & 1u;
      if (!mbar_wait_or_die(&full[s], par, kWaitBudget, &dead, false)) set_error(err, kErrTimeout);
      __syncwarp();
      if (lane < P) mbar_arrive_remote(&pub[s], (uint32_t)lane);
      __syncwarp();
    }
  } else if (tid >= kCons) {
    // ---- producer warp
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t r = (uint32_t)(k / kStages);
      const int64_t row0 = (cl + k * ncl) * TR;
      const int nr = (int)((rows - row0) < TR ? (rows - row0) : TR);
      float *so = dyn + s * slot_floats;
      float *mall = so + TR * D, *lall = mall + P * TRp;
      if (k >= kStages && !mbar_wait_or_die(&cons[s], (r - 1) & 1u, kWaitBudget, &dead, true))
        set_error(err, kErrTimeout);
      if (!ml_bulk) {
        for (int j = lane; j < P * nr; j += 32) {
          const int q = j / nr, i = j - q * nr;
          mall[q * TRp + i] = __ldg(m + (int64_t)q * rows + row0 + i);
          lall[q * TRp + i] = __ldg(l + (int64_t)q * rows + row0 + i);
        }
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t ob = (uint32_t)nr * (uint32_t)D * 4u;
        const uint32_t mb = ml_bulk ? (uint32_t)nr * 4u : 0u;
        mbar_arrive_expect_tx(&full[s], ob + 2u * P * mb);
        bulk_g2s(so, O + ((int64_t)p * rows + row0) * D, ob, &full[s]);
        if (ml_bulk) {
          for (int q = 0; q < P; ++q) {
            bulk_g2s(mall + q * TRp, m + (int64_t)q * rows + row0, mb, &full[s]);
            bulk_g2s(lall + q * TRp, l + (int64_t)q * rows + row0, mb, &full[s]);
          }
        }
      }
      __syncwarp();
    }
  } else {
    // ---- consumers
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t par = (uint32_t)(k / kStages) & 1u;
      const int64_t row0 = (cl + k * ncl) * TR;
      const int nr = (int)((rows - row0) < TR ? (rows - row0) : TR);
      const float *so = dyn + s * slot_floats;
      // pub[s] completes only after this CTA's own full[s] did (its own
      // publisher arrives too), so it also covers the locally staged (m, l)
      if (!mbar_wait_or_die(&pub[s], par, kWaitBudget, &dead, true)) set_error(err, kErrTimeout);
      row_weights<P>(so + TR * D, so + TR * D + P * TRp, TRp, nr, scale_log2e, sw, sinv);
      named_sync(1, kCons);
      fold_band<P>(so, nr, D, sw, sinv, p, out + row0 * D);
      named_sync(1, kCons);
      // every consumer's reads of the peers' slots have returned (their
      // values were consumed before the barrier), so a relaxed arrive is
      // enough to hand the slots back
      if (tid < P) mbar_arrive_remote_relaxed(&cons[s], (uint32_t)tid);
    }
  }
  // terminal: every CTA has finished all its DSMEM reads and remote arrives
  // before any CTA of the cluster exits
  __syncthreads();
  cluster_sync();
}

// ---------------------------------------------------------------------------
// Push variant of the fast path: the reduce-scatter is done by the bulk copy
// engine instead of per-thread DSMEM loads, and the scatter is along rows
// (the slice of a row-major tile that a peer owns is then contiguous).
// CTA p owns rows [p*TS, (p+1)*TS) of every tile, TS = TR / P.  Per tile:
//   producer  stages O_p[tile, :] and the (m, l) of all P partitions
//             (full[s]);
//   pusher    once full[s] completes, copies slice q of its staged tile into
//             CTA q's receive area recv[s][p] for every q (itself included),
//             each copy completing on CTA q's rfull[s] (P arrivals + bytes);
//   consumers once rfull[s] completes, fold their TS rows over the P
//             received partials from local shared memory in rank order,
//             store bf16, then tell every sender (relaxed remote arrive on
//             its cons[s]) that its slice has been used.
// cons[s] completing at a CTA means every destination has received and used
// what it pushed from slot s, so both its staged tile and the peers'
// receive areas for slot s may be refilled.
// Slot layout: stage TR*D | recv P*TS*D | m_all P*TRp | l_all P*TRp.
template <int P>
__global__ void __launch_bounds__(kPipeThreads)
k_combine_push(const float *__restrict__ O, const float *__restrict__ m,
               const float *__restrict__ l, int64_t rows, int D, int TR, float scale_log2e,
               uint16_t *__restrict__ out, int ml_bulk, int *err) {
  pdl_begin();
  extern __shared__ __align__(128) float dyn[];
  __shared__ __align__(8) uint64_t full[kStages], rfull[kStages], cons[kStages];
  __shared__ int dead;
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t p = cluster_ctarank();
  const int64_t cl = cluster_id_x(), ncl = cluster_nid_x();
  const int64_t ntiles = (rows + TR - 1) / TR;
  const int TS = TR / P;
  const int TRp = (TR + 3) & ~3;
  const int slot_floats = 2 * TR * D + 2 * P * TRp;
  float *sw = dyn + kStages * slot_floats;  // [TS][P]
  float *sinv = sw + TS * P;                // [TS]
  if (tid == 0) {
    dead = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&rfull[s], P);
      mbar_init(&cons[s], P);
    }
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every peer's barriers exist before any remote operation

  const int64_t K = (cl < ntiles) ? (ntiles - 1 - cl) / ncl + 1 : 0;
  auto tile_rows_of = [&](int64_t k) {
    const int64_t row0 = (cl + k * ncl) * TR;
    return (int)((rows - row0) < TR ? (rows - row0) : TR);
  };
  auto slice_rows = [&](int nr, int q) {
    const int a = q * TS, b = a + TS < nr ? a + TS : nr;
    return b > a ? b - a : 0;
  };
  if (tid >= kCons + 32) {
    // ---- pusher warp (lane q serves destination q)
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t par = (uint32_t)(k / kStages) & 1u;
      const int nr = tile_rows_of(k);
      float *stage = dyn + s * slot_floats;
      float *recv = stage + TR * D;
      if (!mbar_wait_or_die(&full[s], par, kWaitBudget, &dead, false)) set_error(err, kErrTimeout);
      __syncwarp();
      if (lane < P) {
        const int q = lane;
        const uint32_t bytes = (uint32_t)slice_rows(nr, q) * (uint32_t)D * 4u;
        mbar_arrive_expect_tx_remote(&rfull[s], (uint32_t)q, bytes);
        if (bytes)
          bulk_s2peer(recv + p * TS * D, stage + q * TS * D, bytes, &rfull[s], (uint32_t)q);
      }
      __syncwarp();
    }
  } else if (tid >= kCons) {
    // ---- producer warp
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t r = (uint32_t)(k / kStages);
      const int64_t row0 = (cl + k * ncl) * TR;
      const int nr = tile_rows_of(k);
      float *stage = dyn + s * slot_floats;
      float *mall = stage + 2 * TR * D, *lall = mall + P * TRp;
      if (k >= kStages && !mbar_wait_or_die(&cons[s], (r - 1) & 1u, kWaitBudget, &dead, true))
        set_error(err, kErrTimeout);
      if (!ml_bulk) {
        for (int j = lane; j < P * nr; j += 32) {
          const int q = j / nr, i = j - q * nr;
          mall[q * TRp + i] = __ldg(m + (int64_t)q * rows + row0 + i);
          lall[q * TRp + i] = __ldg(l + (int64_t)q * rows + row0 + i);
        }
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t ob = (uint32_t)nr * (uint32_t)D * 4u;
        const uint32_t mb = ml_bulk ? (uint32_t)nr * 4u : 0u;
        mbar_arrive_expect_tx(&full[s], ob + 2u * P * mb);
        bulk_g2s(stage, O + ((int64_t)p * rows + row0) * D, ob, &full[s]);
        if (ml_bulk) {
          for (int q = 0; q < P; ++q) {
            bulk_g2s(mall + q * TRp, m + (int64_t)q * rows + row0, mb, &full[s]);
            bulk_g2s(lall + q * TRp, l + (int64_t)q * rows + row0, mb, &full[s]);
          }
        }
      }
      __syncwarp();
    }
  } else {
    // ---- consumers: this CTA's TS rows of each tile
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % kStages);
      const uint32_t par = (uint32_t)(k / kStages) & 1u;
      const int64_t row0 = (cl + k * ncl) * TR;
      const int nr = tile_rows_of(k);
      const int ns = slice_rows(nr, (int)p);
      const float *stage = dyn + s * slot_floats;
      const float *recv = stage + TR * D;
      const float *mall = stage + 2 * TR * D, *lall = mall + P * TRp;
      // rfull[s] includes this CTA's own push, issued after its full[s]
      // completed, so the staged (m, l) are covered too
      if (!mbar_wait_or_die(&rfull[s], par, kWaitBudget, &dead, true)) set_error(err, kErrTimeout);
      const int i0 = (int)p * TS;
      for (int i = tid; i < ns; i += kCons) {
        float mq[P];
#pragma unroll
        for (int q = 0; q < P; ++q) mq[q] = mall[q * TRp + i0 + i];
        float M = mq[0];
#pragma unroll
        for (int q = 1; q < P; ++q) M = fmaxf(M, mq[q]);
        float L = 0.0f;
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float w = (M == -INFINITY) ? 0.0f : ex2f_approx((mq[q] - M) * scale_log2e);
          sw[i * P + q] = w;
          L = fmaf(w, lall[q * TRp + i0 + i], L);
        }
        sinv[i] = (M == -INFINITY || L == 0.0f) ? 0.0f : 1.0f / L;
      }
      named_sync(1, kCons);
      const int cpr = D >> 2;
      for (int c = tid; c < ns * cpr; c += kCons) {
        const int i = c / cpr, col = 4 * (c - i * cpr);
        float4 v[P];
#pragma unroll
        for (int q = 0; q < P; ++q)
          v[q] = *reinterpret_cast<const float4 *>(recv + (q * TS + i) * D + col);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float w = sw[i * P + q];
          acc.x = fmaf(w, v[q].x, acc.x);
          acc.y = fmaf(w, v[q].y, acc.y);
          acc.z = fmaf(w, v[q].z, acc.z);
          acc.w = fmaf(w, v[q].w, acc.w);
        }
        const float inv = sinv[i];
        uint2 pk = make_uint2(0u, 0u);
        if (inv != 0.0f) {
          pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        }
        *reinterpret_cast<uint2 *>(out + (row0 + i0 + i) * D + col) = pk;
      }
      named_sync(1, kCons);
      if (tid < P) mbar_arrive_remote_relaxed(&cons[s], (uint32_t)tid);
    }
  }
  __syncthreads();
  cluster_sync();
}

// ---------------------------------------------------------------------------
// Direct variant: no exchange between CTAs at all.  Each CTA streams tiles
// of TR rows, staging the rows of all P partitions (P contiguous 1-D bulk
// copies; the (m, l) by the producer warp) through a ring of S slots,
// then folds every row over the P partials in rank order from local shared
// memory.  DRAM traffic is the same as the cluster variants' (each partial
// byte is read once); what it drops is the per-tile cluster synchronisation.
// Slot layout: O_all P*TR*D | m_all P*TRp | l_all P*TRp.
//   full[s]  (local, 1 arrival + tx)  the slot's copies and loads landed;
//   free[s]  (local, 1 arrival)       the consumers are done with the slot.
// Held to 8 CTAs per SM (40 registers at 192 threads): the overlap of this
// variant comes from the other CTAs on the SM, and the compiler's own
// choice for P = 8 went to 56 registers and 5 CTAs.
template <int P, int S>
__global__ void __launch_bounds__(kPipeThreads, 8)
k_combine_direct(const float *__restrict__ O, const float *__restrict__ m,
                 const float *__restrict__ l, int64_t rows, int D, int TR, float scale_log2e,
                 uint16_t *__restrict__ out, int ml_bulk, int *err) {
  pdl_begin();
  extern __shared__ __align__(128) float dyn[];
  __shared__ __align__(8) uint64_t full[S], freed[S];
  __shared__ int dead;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t ntiles = (rows + TR - 1) / TR;
  const int TRp = (TR + 3) & ~3;
  const int slot_floats = P * TR * D + 2 * P * TRp;
  float *sw = dyn + S * slot_floats;  // [TR][P]
  float *sinv = sw + TR * P;                // [TR]
  if (tid == 0) {
    dead = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&freed[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t K = ((int64_t)blockIdx.x < ntiles) ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (tid >= kCons + 32) {
    // idle warp (keeps the block shape of the cluster variants)
  } else if (tid >= kCons) {
    // ---- producer warp
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % S);
      const uint32_t r = (uint32_t)(k / S);
      const int64_t row0 = ((int64_t)blockIdx.x + k * gridDim.x) * TR;
      const int nr = (int)((rows - row0) < TR ? (rows - row0) : TR);
      float *so = dyn + s * slot_floats;
      float *mall = so + P * TR * D, *lall = mall + P * TRp;
      if (k >= S &&
          !mbar_wait_or_die(&freed[s], (r - 1) & 1u, kWaitBudget, &dead, false))
        set_error(err, kErrTimeout);
      // arm the byte count and start the big copies first, then fetch the
      // (m, l) while they fly (with ml_bulk they ride the copy engine too:
      // fetched by the lanes, two dependent round trips per tile for P * TR
      // > 32 sat on the critical path of small tiles); the arrival releases
      // the (m, l) stores
      if (lane == 0) {
        const uint32_t ob = (uint32_t)nr * (uint32_t)D * 4u;
        const uint32_t mb = ml_bulk ? (uint32_t)nr * 4u : 0u;
        mbar_expect_tx(&full[s], ob * P + 2u * P * mb);
        for (int q = 0; q < P; ++q)
          bulk_g2s(so + q * TR * D, O + ((int64_t)q * rows + row0) * D, ob, &full[s]);
        if (ml_bulk) {
          for (int q = 0; q < P; ++q) {
            bulk_g2s(mall + q * TRp, m + (int64_t)q * rows + row0, mb, &full[s]);
            bulk_g2s(lall + q * TRp, l + (int64_t)q * rows + row0, mb, &full[s]);
          }
        }
      }
      if (!ml_bulk) {
        for (int j = lane; j < P * nr; j += 32) {
          const int q = j / nr, i = j - q * nr;
          mall[q * TRp + i] = __ldg(m + (int64_t)q * rows + row0 + i);
          lall[q * TRp + i] = __ldg(l + (int64_t)q * rows + row0 + i);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
      __syncwarp();
    }
  } else {
    // ---- consumers
    for (int64_t k = 0; k < K; ++k) {
      const int s = (int)(k % S);
      const uint32_t par = (uint32_t)(k / S) & 1u;
      const int64_t row0 = ((int64_t)blockIdx.x + k * gridDim.x) * TR;
      const int nr = (int)((rows - row0) < TR ? (rows - row0) : TR);
      const float *so = dyn + s * slot_floats;
      const float *mall = so + P * TR * D, *lall = mall + P * TRp;
      if (!mbar_wait_or_die(&full[s], par, kWaitBudget, &dead, false)) set_error(err, kErrTimeout);
      for (int i = tid; i < nr; i += kCons) {
        float mq[P];
#pragma unroll
        for (int q = 0; q < P; ++q) mq[q] = mall[q * TRp + i];
        float M = mq[0];
#pragma unroll
        for (int q = 1; q < P; ++q) M = fmaxf(M, mq[q]);
        float L = 0.0f;
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float w = (M == -INFINITY) ? 0.0f : ex2f_approx((mq[q] - M) * scale_log2e);
          sw[i * P + q] = w;
          L = fmaf(w, lall[q * TRp + i], L);
        }
        sinv[i] = (M == -INFINITY || L == 0.0f) ? 0.0f : 1.0f / L;
      }
      named_sync(1, kCons);
      const int cpr = D >> 2;
      for (int c = tid; c < nr * cpr; c += kCons) {
        const int i = c / cpr, col = 4 * (c - i * cpr);
        float4 v[P];
#pragma unroll
        for (int q = 0; q < P; ++q)
          v[q] = *reinterpret_cast<const float4 *>(so + (q * TR + i) * D + col);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < P; ++q) {
          const float w = sw[i * P + q];
          acc.x = fmaf(w, v[q].x, acc.x);
          acc.y = fmaf(w, v[q].y, acc.y);
          acc.z = fmaf(w, v[q].z, acc.z);
          acc.w = fmaf(w, v[q].w, acc.w);
        }
        const float inv = sinv[i];
        uint2 pk = make_uint2(0u, 0u);
        if (inv != 0.0f) {
          pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        }
        *reinterpret_cast<uint2 *>(out + (row0 + i) * D + col) = pk;
      }
      named_sync(1, kCons);
      if (tid == 0) mbar_arrive(&freed[s]);
    }
  }
  __syncthreads();
}

// Generic path: one tile per cluster, plain loads, per-element bands.
__global__ void __launch_bounds__(kCombThreads)
k_combine_generic(const float *__restrict__ O, const float *__restrict__ m,
                  const float *__restrict__ l, int64_t rows, int D, int TR, float scale_log2e,
                  uint16_t *__restrict__ out) {
  pdl_begin();
  extern __shared__ __align__(128) float dyn[];
  const int tid = threadIdx.x;
  const uint32_t P = cluster_nctarank(), p = cluster_ctarank();
  const int64_t row0 = (int64_t)cluster_id_x() * TR;
  const int nr = (int)((rows - row0) < TR ? (rows - row0) : TR);
  float *sO = dyn;
  float *sm = sO + TR * D;
  float *sl = sm + TR;
  float *sw = sl + TR;
  float *sinv = sw + TR * P;
  const float *Op = O + ((int64_t)p * rows + row0) * D;
  for (int i = tid; i < nr * D; i += kCombThreads) sO[i] = __ldg(Op + i);
  for (int i = tid; i < nr; i += kCombThreads) {
    sm[i] = __ldg(m + (int64_t)p * rows + row0 + i);
    sl[i] = __ldg(l + (int64_t)p * rows + row0 + i);
  }
  cluster_sync();  // publish, every partition, band or not
  for (int i = tid; i < nr; i += kCombThreads) {
    const uint32_t am = smem_u32(sm + i), al = smem_u32(sl + i);
    float M = -INFINITY;
    for (uint32_t q = 0; q < P; ++q) M = fmaxf(M, ld_dsmem_f32(map_peer(am, q)));
    float L = 0.0f;
    for (uint32_t q = 0; q < P; ++q) {
      const float w = (M == -INFINITY) ? 0.0f
                                       : ex2f_approx((ld_dsmem_f32(map_peer(am, q)) - M) * scale_log2e);
      sw[i * P + q] = w;
      L = fmaf(w, ld_dsmem_f32(map_peer(al, q)), L);
    }
    sinv[i] = (M == -INFINITY || L == 0.0f) ? 0.0f : 1.0f / L;
  }
  __syncthreads();
  const int b0 = (int)((int64_t)p * D / P), b1 = (int)((int64_t)(p + 1) * D / P);
  const int bw = b1 - b0;
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
  cluster_sync();  // terminal
}

int tile_rows(int64_t rows, int D) {
  int TR = kTileBytes / (D * 4);
  if (TR < 1) TR = 1;
  if (TR > 64) TR = 64;
  if (TR >= 4) TR &= ~3;
  if ((int64_t)TR > rows) TR = (int)rows;
  return TR;
}

template <class K>
int prepare(K kern, int P, size_t smem) {
  cudaError_t e;
  if (P > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return RR_OK;
}

template <int P>
int launch_pipe(const float *O, const float *m, const float *l, int64_t rows, int D,
                float scale_log2e, uint16_t *out, cudaStream_t s, const DevInfo &d) {
  const int TR = tile_rows(rows, D);
  const size_t TRp = ((size_t)TR + 3) & ~(size_t)3;
  const size_t smem = sizeof(float) * ((size_t)kStages * ((size_t)TR * D + 2 * P * TRp) +
                                       (size_t)TR * P + (size_t)TR);
  auto kern = k_combine_pipe<P>;
  int st = prepare(kern, P, smem);
  if (st != RR_OK) return st;
  const int64_t ntiles = (rows + TR - 1) / TR;
  int clusters = 1;
  {
    const int n = occupancy_clusters((const void *)kern, kPipeThreads, smem, P, d.device);
    if (n < 1) return RR_ERR_UNSUPPORTED;
    clusters = n;
  }
  if ((int64_t)clusters > ntiles) clusters = (int)ntiles;
  const int ml_bulk = (rows % 4 == 0) && (TR % 4 == 0) && ((uintptr_t)m % 16 == 0) &&
                      ((uintptr_t)l % 16 == 0);
  if (log_enabled())
    std::fprintf(stderr, "rr: combine pipe P=%d D=%d TR=%d stages=%d clusters=%d smem=%zu ml_bulk=%d\n",
                 P, D, TR, kStages, clusters, smem, ml_bulk);
  return cuda_status(launch_kernel(kern, dim3((unsigned)(clusters * P)), dim3(kPipeThreads), smem, s, P,
                                   O, m, l, rows, D, TR, scale_log2e, out, ml_bulk, d.err_word));
}

template <int P>
int launch_push(const float *O, const float *m, const float *l, int64_t rows, int D,
                float scale_log2e, uint16_t *out, cudaStream_t s, const DevInfo &d) {
  // tile rows: a multiple of max(P, 4), at least P (a tile may overrun rows)
  const int unit = P > 4 ? P : 4;
  int TR = kTileBytes / (D * 4);
  TR = (TR / unit) * unit;
  if (TR < unit) TR = unit;
  const int TS = TR / P;
  const size_t TRp = ((size_t)TR + 3) & ~(size_t)3;
  const size_t smem = sizeof(float) * ((size_t)kStages * (2 * (size_t)TR * D + 2 * P * TRp) +
                                       (size_t)TS * P + (size_t)TS);
  auto kern = k_combine_push<P>;
  int st = prepare(kern, P, smem);
  if (st != RR_OK) return st;
  const int64_t ntiles = (rows + TR - 1) / TR;
  int clusters = 1;
  {
    const int n = occupancy_clusters((const void *)kern, kPipeThreads, smem, P, d.device);
    if (n < 1) return RR_ERR_UNSUPPORTED;
    clusters = n;
  }
  if ((int64_t)clusters > ntiles) clusters = (int)ntiles;
  const int ml_bulk = (rows % 4 == 0) && ((uintptr_t)m % 16 == 0) && ((uintptr_t)l % 16 == 0);
  if (log_enabled())
    std::fprintf(stderr, "rr: combine push P=%d D=%d TR=%d stages=%d clusters=%d smem=%zu ml_bulk=%d\n",
                 P, D, TR, kStages, clusters, smem, ml_bulk);
  return cuda_status(launch_kernel(kern, dim3((unsigned)(clusters * P)), dim3(kPipeThreads), smem, s, P,
                                   O, m, l, rows, D, TR, scale_log2e, out, ml_bulk, d.err_word));
}

// Direct variant geometry, from sweeps on GB300 (256 MiB of partials, D =
// 64, 128, 256, and the 131072 x 128 workloads): tiles of 16 KiB for
// P <= 8, 32 KiB for P = 16.  The (m, l) of a tile go by the copy engine
// when the producer's lanes would need more than one round trip for them
// (more than 32 (partition, row) pairs; every tile 16-byte aligned): two
// dependent round trips sat on the critical path of small tiles (D = 64 ran
// at 0.66-0.80 of the copy bandwidth for P = 4..16), while for 32 pairs or
// fewer the copies only add work (P = 8, D = 128: 0.96 against 0.98).  One
// slot per CTA (the other CTAs on the SM provide the overlap), two for
// P = 16 and for P = 8 with copied (m, l).
#ifndef RR_DIRECT_BYTES
#define RR_DIRECT_BYTES 16384
#endif

template <int P, int S>
int launch_direct_s(const float *O, const float *m, const float *l, int64_t rows, int D, int TR,
                    int ml_bulk, float scale_log2e, uint16_t *out, cudaStream_t s,
                    const DevInfo &d) {
  const size_t TRp = ((size_t)TR + 3) & ~(size_t)3;
  const size_t smem = sizeof(float) * ((size_t)S * ((size_t)P * TR * D + 2 * P * TRp) +
                                       (size_t)TR * P + (size_t)TR);
  auto kern = k_combine_direct<P, S>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const int nb = occupancy_blocks((const void *)kern, kPipeThreads, smem, d.device);
  const int64_t ntiles = (rows + TR - 1) / TR;
  int64_t grid = (int64_t)nb * d.sm_count;
  if (grid > ntiles) grid = ntiles;
  if (log_enabled())
    std::fprintf(stderr, "rr: combine direct P=%d D=%d TR=%d stages=%d ctas=%lld smem=%zu ml_bulk=%d\n",
                 P, D, TR, S, (long long)grid, smem, ml_bulk);
  launch_kernel(kern, dim3((unsigned)grid), dim3(kPipeThreads), smem, s, 0, O, m, l, rows, D, TR,
                scale_log2e, out, ml_bulk, d.err_word);
  return cuda_status(cudaGetLastError());
}

template <int P>
int launch_direct(const float *O, const float *m, const float *l, int64_t rows, int D,
                  float scale_log2e, uint16_t *out, cudaStream_t s, const DevInfo &d) {
  const int bytes = P <= 8 ? RR_DIRECT_BYTES : 32768;
  int TR = bytes / (P * D * 4);
  if (TR < 1) TR = 1;
  if ((int64_t)TR > rows) TR = (int)rows;
  const int ml_bulk = (P * TR > 32) && (rows % 4 == 0) && (TR % 4 == 0) &&
                      ((uintptr_t)m % 16 == 0) && ((uintptr_t)l % 16 == 0);
  if constexpr (P == 16) {
    return launch_direct_s<P, 2>(O, m, l, rows, D, TR, ml_bulk, scale_log2e, out, s, d);
  } else if constexpr (P == 8) {
    if (ml_bulk) return launch_direct_s<P, 2>(O, m, l, rows, D, TR, ml_bulk, scale_log2e, out, s, d);
    return launch_direct_s<P, 1>(O, m, l, rows, D, TR, ml_bulk, scale_log2e, out, s, d);
  } else {
    return launch_direct_s<P, 1>(O, m, l, rows, D, TR, ml_bulk, scale_log2e, out, s, d);
  }
}

int launch_generic(const float *O, const float *m, const float *l, int P, int64_t rows, int D,
                   float scale_log2e, uint16_t *out, cudaStream_t s) {
  const int TR = tile_rows(rows, D);
  const size_t smem = sizeof(float) * ((size_t)TR * D + 2 * (size_t)TR + (size_t)TR * P + TR);
  int st = prepare(k_combine_generic, P, smem);
  if (st != RR_OK) return st;
  const int64_t tiles = (rows + TR - 1) / TR;
  if (tiles * P > 0x7fffffffLL) return RR_ERR_INVALID;
  int dev = 0;
  if (P > 1 && (cudaGetDevice(&dev) != cudaSuccess ||
                occupancy_clusters((const void *)k_combine_generic, kCombThreads, smem, P, dev) < 1)) {
    cudaGetLastError();
    return RR_ERR_UNSUPPORTED;
  }
  if (log_enabled())
    std::fprintf(stderr, "rr: combine generic P=%d D=%d TR=%d clusters=%lld smem=%zu\n", P, D, TR,
                 (long long)tiles, smem);
  return cuda_status(launch_kernel(k_combine_generic, dim3((unsigned)(tiles * P)), dim3(kCombThreads),
                                   smem, s, P, O, m, l, rows, D, TR, scale_log2e, out));
}

}  // namespace

int launch_combine(const float *O, const float *m, const float *l, int P, int64_t rows, int D,
                   float scale_log2e, uint16_t *out, cudaStream_t s, const DevInfo &d, int mode) {
  const bool pow2 = (P == 1 || P == 2 || P == 4 || P == 8 || P == 16);
  const bool aligned = ((uintptr_t)O % 16 == 0) && ((uintptr_t)out % 8 == 0);
  const bool pull_ok = pow2 && D % (4 * P) == 0 && aligned;
  const bool push_ok = pow2 && D % 4 == 0 && aligned && D <= 256;
  const bool direct_ok = pow2 && D % 4 == 0 && aligned && (size_t)2 * P * D * 4 <= (size_t)96 * 1024;
  if (mode == RR_COMBINE_AUTO)
    mode = direct_ok ? RR_COMBINE_DIRECT
                     : (push_ok ? RR_COMBINE_PUSH : (pull_ok ? RR_COMBINE_PULL : RR_COMBINE_GENERIC));
  if (mode == RR_COMBINE_DIRECT) {
    if (!direct_ok) return RR_ERR_UNSUPPORTED;
    switch (P) {
      case 1: return launch_direct<1>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 2: return launch_direct<2>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 4: return launch_direct<4>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 8: return launch_direct<8>(O, m, l, rows, D, scale_log2e, out, s, d);
      default: return launch_direct<16>(O, m, l, rows, D, scale_log2e, out, s, d);
    }
  }
  // the remaining variants exchange through a cluster of P CTAs
  if (P > 1 && !d.cluster_launch) return RR_ERR_UNSUPPORTED;
  if (mode == RR_COMBINE_PUSH) {
    if (!push_ok) return RR_ERR_UNSUPPORTED;
    switch (P) {
      case 1: return launch_push<1>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 2: return launch_push<2>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 4: return launch_push<4>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 8: return launch_push<8>(O, m, l, rows, D, scale_log2e, out, s, d);
      default: return launch_push<16>(O, m, l, rows, D, scale_log2e, out, s, d);
    }
  }
  if (mode == RR_COMBINE_PULL) {
    if (!pull_ok) return RR_ERR_UNSUPPORTED;
    switch (P) {
      case 1: return launch_pipe<1>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 2: return launch_pipe<2>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 4: return launch_pipe<4>(O, m, l, rows, D, scale_log2e, out, s, d);
      case 8: return launch_pipe<8>(O, m, l, rows, D, scale_log2e, out, s, d);
      default: return launch_pipe<16>(O, m, l, rows, D, scale_log2e, out, s, d);
    }
  }
  return launch_generic(O, m, l, P, rows, D, scale_log2e, out, s);
}

}  // namespace rr
