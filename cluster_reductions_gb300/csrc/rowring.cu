// rowring.cu -- the two-pass row operations of the "reduce" page
// (algorithm/gpu/rowwise: softmax, layernorm statistics, layernorm rewrite)
// for long rows, streamed through a ring of shared-memory slots filled by
// the bulk copy engine.
//
// Persistent clusters of C CTAs (C = 1: a CTA per row); cluster k takes rows
// k, k + nclusters, ...  and CTA r of the cluster owns the slice
// [r * chunk, min((r + 1) * chunk, cols)) of each of them (chunk a multiple
// of 8 elements, so every slice starts 16-byte aligned when the row does).
// The CTA's work is a sequence of pieces of its slices (6 or 12 KiB each),
// row by row and pass by pass; piece i belongs to consumer warp i % 8, which
// owns two ring slots: it bulk-copies its pieces into them two ahead, folds
// (or rewrites) each piece as it lands and, once done with a slot, starts
// the copy of its piece i + 16 there -- across passes and rows, since no
// copy depends on a result.
//
// Each row takes ONE combine over the cluster, of a monoid state:
//   softmax     the online (max, sum) pair;
//   layernorm   (count, mean, M2), M2 the sum of squared deviations from the
//               mean, merged with the update of Chan, Golub and LeVeque
//               ("Updating formulae and a pairwise algorithm for computing
//               sample variances", 1979): n = na + nb, d = mean_b - mean_a,
//               mean = mean_a + d nb / n, M2 = M2a + M2b + d^2 na nb / n.
//               Every leaf is the slots a thread holds of one piece, folded
//               two-pass about the leaf's own mean, so the variance is
//               computed about means at every level (never E[x^2] - mean^2)
//               and the row is read once.
// The combine ("cluster_allreduce" page: every CTA gathers every peer's
// value and folds them in rank order, so all CTAs hold the same bits) is
// done with remote stores instead of a cluster barrier, so that only one
// thread (the reducer) takes part in it: that thread of every CTA writes its state
// into slot [row parity][its rank] of every peer and arrives (release,
// cluster scope) on that peer's mbarrier of the same parity; each CTA waits
// for C arrivals and folds slots 0..C-1 in rank order.  Two parities
// alternate over the rows, as the page's two-slot form does: a CTA can
// write a parity again (two rows later) only after every peer has sent the
// next row's state, which each sends after it has folded this parity.
// The second pass of softmax and of the rewrite streams the slice again
// (from L2: the plan takes this kernel for them only while the rows in
// flight fit it), with the outputs computed from the ring.
#include <cstdio>

#include "rr.h"
#include "rr_device.cuh"
#include "rr_internal.h"
#include "rowwise.cuh"

namespace rr {
namespace {

constexpr int kRingConsWarps = 8;             // consumer warps
constexpr int kRingThreads = (kRingConsWarps + 1) * 32;  // + the reducer warp
// Ring slots: item i (a piece) goes to slot i % kRingStages and to consumer
// warp i % kRingConsWarps.  With the slot count a multiple of the warp count
// every slot belongs to one warp, which fills it and waits on each phase of
// its full barrier in order: a parity wait can only tell the awaited phase
// from the one before it, so a warp that skipped phases of a slot could
// take the previous phase's completion for the one it waits for.
constexpr int kRingStages = 16;
static_assert(kRingStages % kRingConsWarps == 0, "one consumer warp per slot");
// Bytes per slot and bulk copy: 12 KiB with one CTA per SM (192 KiB of
// slots), 6 KiB with two.  Either splits into whole leaves of 3 units
// (8 elements each) a lane: 96 units per leaf round of a warp.
constexpr uint32_t kRingPieceBig = 12288, kRingPieceSmall = 6144;

// 8 elements (a "unit": 16 bytes of bf16, 32 bytes of fp32) of a ring slot.
template <class In>
__device__ __forceinline__ void ring_unit(const unsigned char *slot, int u, float (&e)[8]) {
  if constexpr (In::EPV == 8) {
    In::unpack(*reinterpret_cast<const uint4 *>(slot + (size_t)u * 16), e);
  } else {
    const uint4 a = *reinterpret_cast<const uint4 *>(slot + (size_t)u * 32);
    const uint4 b = *reinterpret_cast<const uint4 *>(slot + (size_t)u * 32 + 16);
    e[0] = __uint_as_float(a.x); e[1] = __uint_as_float(a.y);
    e[2] = __uint_as_float(a.z); e[3] = __uint_as_float(a.w);
    e[4] = __uint_as_float(b.x); e[5] = __uint_as_float(b.y);
    e[6] = __uint_as_float(b.z); e[7] = __uint_as_float(b.w);
  }
}

// The same unit as four packed fp32 pairs (elements 2k, 2k + 1 in pair k).
template <class In>
__device__ __forceinline__ void ring_unit2(const unsigned char *slot, int u, uint64_t (&p)[4]) {
  if constexpr (In::EPV == 8) {
    const uint4 w = *reinterpret_cast<const uint4 *>(slot + (size_t)u * 16);
    p[0] = bf16x2_to_f2(w.x);
    p[1] = bf16x2_to_f2(w.y);
    p[2] = bf16x2_to_f2(w.z);
    p[3] = bf16x2_to_f2(w.w);
  } else {
    const uint4 a = *reinterpret_cast<const uint4 *>(slot + (size_t)u * 32);
    const uint4 b = *reinterpret_cast<const uint4 *>(slot + (size_t)u * 32 + 16);
    p[0] = ((uint64_t)a.y << 32) | a.x;
    p[1] = ((uint64_t)a.w << 32) | a.z;
    p[2] = ((uint64_t)b.y << 32) | b.x;
    p[3] = ((uint64_t)b.w << 32) | b.z;
  }
}

// MODE kModeSoftmax: y (fp32); kModeStats: mean, rstd; kModeLayernorm: ybf
// (bf16), mean / rstd optional.  Requires x 16-byte aligned and cols a
// multiple of 8; y 32-byte aligned (softmax); ybf 16-byte and gamma / beta
// 16-byte aligned (rewrite); chunk a multiple of 8 with chunk * element size
// < 2^32; kRingStages slots of `piece` bytes (a multiple of 32) of dynamic
// shared memory.
//
// Warps: 0..kRingConsWarps-1 stream and consume, the last one reduces.  The
// CTA's work is a sequence of items -- for each of its rows, for each pass,
// the pieces of its slice in order -- and item i belongs to consumer warp
// i % kRingConsWarps, which copies it into its slot i % kRingStages, folds
// (or, in the second pass, rewrites) the whole piece, then starts the copy
// of its item i + kRingStages into the same slot.  At the end of a
// row's first pass every consumer warp reduces its lanes (an xor butterfly,
// the lower lane always the left operand) and leaves its state in wst[row
// parity][warp]; the reducer folds the warps' states in warp order, does
// the cluster exchange, computes the row's result, writes the statistics
// and publishes the result for the second pass, so that the consumers never
// wait at the end of a row unless they need its result.
template <class In, int MODE>
__global__ void __launch_bounds__(kRingThreads, MODE == kModeStats ? 2 : 1)
k_rowwise_ring(const typename In::S *__restrict__ x, int64_t rows, int64_t cols, int64_t chunk,
               uint32_t piece, float eps, float *__restrict__ y, float *__restrict__ mean,
               float *__restrict__ rstd, const float *__restrict__ gamma,
               const float *__restrict__ beta, uint16_t *__restrict__ ybf, int *err) {
  pdl_begin();
  using S = typename In::S;
  constexpr int E = (int)sizeof(S);
  constexpr int NW = kRingConsWarps;
  constexpr int NPASS = MODE == kModeStats ? 1 : 2;
  constexpr int UB = 8 * E;                    // bytes per unit (8 elements)
  constexpr int LEAF = 4;                      // units per lane and leaf
  constexpr uint32_t stages = kRingStages;
  const int UPP = (int)(piece / UB);           // units per whole piece
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kRingStages];
  __shared__ __align__(8) uint64_t xbar[2], rowbar[2], rowres[2];
  __shared__ __align__(16) uint32_t xslot[2][16][4];
  __shared__ __align__(16) uint32_t wst[2][NW][4];
  __shared__ float res[2][4];
  __shared__ int dead;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank(), r = cluster_ctarank();
  const int64_t cl = cluster_id_x(), ncl = cluster_nid_x();
  const int64_t b0 = (int64_t)r * chunk < cols ? (int64_t)r * chunk : cols;
  const int64_t b1 = b0 + chunk < cols ? b0 + chunk : cols;
  const uint32_t bytes = (uint32_t)((b1 - b0) * E);  // a multiple of UB
  const int np = (int)((bytes + piece - 1) / piece);
  const int64_t nrow = cl < rows ? (rows - 1 - cl) / ncl + 1 : 0;  // rows of this cluster

  if (tid == 0) {
    dead = 0;
    for (int s = 0; s < kRingStages; ++s) mbar_init(&full[s], 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&xbar[k], C);
      mbar_init(&rowbar[k], NW);
      mbar_init(&rowres[k], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (C > 1) cluster_sync();  // every peer's xbar exists before any remote arrive

  // units (8 elements) in piece p of the slice
  auto piece_units = [&](int p) -> int {
    const uint32_t off = (uint32_t)p * piece;
    return (int)((bytes - off < piece ? bytes - off : piece) / UB);
  };
  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (!mbar_wait_or_die(bar, parity, kWaitBudget, &dead, false)) set_error(err, kErrTimeout);
  };

  // item i: piece i % np of pass (i / np) % NPASS of the CTA's row i / (NPASS np)
  const uint32_t per_row = (uint32_t)(NPASS * np);
  const uint32_t total = (uint32_t)nrow * per_row;
  auto issue = [&](uint32_t item) {  // one lane: copy item into its slot
    const uint32_t jj = item / per_row, p = (item - jj * per_row) % (uint32_t)np;
    const unsigned char *src =
        reinterpret_cast<const unsigned char *>(x + (cl + (int64_t)jj * ncl) * cols + b0);
    const uint32_t off = p * piece;
    const uint32_t len = bytes - off < piece ? bytes - off : piece;
    const int s = (int)(item % stages);
    // the warp's earlier reads of the slot (generic proxy) come before the
    // copy engine's writes into it (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(&full[s], len);
    bulk_g2s(ring + (size_t)s * piece, src + off, len, &full[s]);
  };

  if (warp == NW) {
    // ---- reducer: per row, the warps' states in warp order, then the
    // cluster in rank order
    if (lane == 0) {
      for (int64_t j = 0; j < nrow; ++j) {
        const int64_t row = cl + j * ncl;
        const uint32_t par = (uint32_t)(j & 1), ph = (uint32_t)(j >> 1) & 1u;
        wait(&rowbar[par], ph);
        uint4 w;
        if constexpr (MODE == kModeSoftmax) {
          float m = __uint_as_float(wst[par][0][0]), sm = __uint_as_float(wst[par][0][1]);
          for (int k = 1; k < NW; ++k)
            ms_combine(m, sm, __uint_as_float(wst[par][k][0]), __uint_as_float(wst[par][k][1]));
          w = make_uint4(__float_as_uint(m), __float_as_uint(sm), 0u, 0u);
        } else {
          Chan t{wst[par][0][0], __uint_as_float(wst[par][0][1]), __uint_as_float(wst[par][0][2])};
          for (int k = 1; k < NW; ++k)
            t = chan_merge(t, Chan{wst[par][k][0], __uint_as_float(wst[par][k][1]),
                                   __uint_as_float(wst[par][k][2])});
          w = make_uint4(t.n, __float_as_uint(t.mean), __float_as_uint(t.m2), 0u);
        }
        if (C > 1) {
          // every CTA's state into slot [parity][rank] of every peer, then
          // an arrive (release, cluster scope) on that peer's xbar
          const uint32_t a = smem_u32(&xslot[par][r][0]);
          for (uint32_t q = 0; q < C; ++q) {
            st_dsmem_u4(map_peer(a, q), w);
            mbar_arrive_remote(&xbar[par], q);
          }
          if (!mbar_wait_or_die(&xbar[par], ph, kWaitBudget, &dead, true))
            set_error(err, kErrTimeout);
          if constexpr (MODE == kModeSoftmax) {
            float m = __uint_as_float(xslot[par][0][0]), sm = __uint_as_float(xslot[par][0][1]);
            for (uint32_t q = 1; q < C; ++q)
              ms_combine(m, sm, __uint_as_float(xslot[par][q][0]),
                         __uint_as_float(xslot[par][q][1]));
            w = make_uint4(__float_as_uint(m), __float_as_uint(sm), 0u, 0u);
          } else {
            Chan t{xslot[par][0][0], __uint_as_float(xslot[par][0][1]),
                   __uint_as_float(xslot[par][0][2])};
            for (uint32_t q = 1; q < C; ++q)
              t = chan_merge(t, Chan{xslot[par][q][0], __uint_as_float(xslot[par][q][1]),
                                     __uint_as_float(xslot[par][q][2])});
            w = make_uint4(t.n, __float_as_uint(t.mean), __float_as_uint(t.m2), 0u);
          }
        }
        if constexpr (MODE == kModeSoftmax) {
          res[par][0] = __uint_as_float(w.x);
          res[par][1] = 1.0f / __uint_as_float(w.y);
        } else {
          const float mu = __uint_as_float(w.y);
          const float rs = 1.0f / sqrtf(__uint_as_float(w.z) / (float)cols + eps);
          res[par][0] = mu;
          res[par][1] = rs;
          if (r == 0) {
            if (mean) mean[row] = mu;
            if (rstd) rstd[row] = rs;
          }
        }
        mbar_arrive(&rowres[par]);
      }
    }
  } else {
    // ---- consumer warp `warp`: its first two items into its two slots
    if (lane == 0) {
      if ((uint32_t)warp < total) issue((uint32_t)warp);
      if ((uint32_t)(warp + NW) < total) issue((uint32_t)(warp + NW));
    }
    uint32_t it = 0;
    for (int64_t j = 0; j < nrow; ++j) {
      const int64_t row = cl + j * ncl;
      const uint32_t par = (uint32_t)(j & 1), ph = (uint32_t)(j >> 1) & 1u;
      // ---- pass 1: this warp's pieces of the row into its lanes' states
      float m = -INFINITY, sm = 0.0f;  // softmax
      Chan st{0u, 0.0f, 0.0f};         // layernorm
      for (int p = 0; p < np; ++p, ++it) {
        if ((int)(it % (uint32_t)NW) != warp) continue;
        const int s = (int)(it % stages);
        wait(&full[s], (it / stages) & 1u);
        const unsigned char *slot = ring + (size_t)s * piece;
        const int nu = piece_units(p);
        if (nu == UPP) {
          // a whole piece: leaves of 3 units a lane (units l*96 + lane +
          // 32k), no predicates
          const int nleaf = UPP / 96;
          if constexpr (MODE == kModeSoftmax) {
            const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
            for (int l = 0; l < nleaf; ++l) {
              uint64_t e2[3][4];
#pragma unroll
              for (int k = 0; k < 3; ++k) ring_unit2<In>(slot, l * 96 + lane + 32 * k, e2[k]);
              // the online update ("reduce" page, softmax pass 1): the
              // running maximum first, then the leaf's terms against it
              float cm = -INFINITY;
#pragma unroll
              for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float lo, hi;
                  f2_unpack(e2[k][q], lo, hi);
                  cm = fmaxf(cm, fmaxf(lo, hi));
                }
              if (cm > m) {
                sm = (m == -INFINITY) ? 0.0f : sm * ex2_approx((m - cm) * kLog2e);
                m = cm;
              }
              if (m != -INFINITY) {
                const uint64_t nmb2 = f2_pack(-m * kLog2e, -m * kLog2e);
                uint64_t aa = 0, ab = 0;
#pragma unroll
                for (int k = 0; k < 3; ++k)
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    float lo, hi;
                    f2_unpack(f2_fma(e2[k][q], l2e2, nmb2), lo, hi);
                    const uint64_t t = f2_pack(ex2_approx(lo), ex2_approx(hi));
                    if (q & 1) ab = f2_add(ab, t); else aa = f2_add(aa, t);
                  }
                float alo, ahi;
                f2_unpack(f2_add(aa, ab), alo, ahi);
                sm += alo + ahi;
              }
            }
          } else {
            // each leaf two-pass about its mean; the leaves of the piece
            // merged in order with exact-count weights (leaf l joins l
            // leaves of the same size: weight 1 / (l + 1), cross term
            // d^2 * 24 l / (l + 1)), then the piece into the lane's state
            Chan pst{0u, 0.0f, 0.0f};
            for (int l = 0; l < nleaf; ++l) {
              uint64_t e2[3][4];
#pragma unroll
              for (int k = 0; k < 3; ++k) ring_unit2<In>(slot, l * 96 + lane + 32 * k, e2[k]);
              uint64_t sa = f2_add(e2[0][0], e2[0][1]), sb = f2_add(e2[0][2], e2[0][3]);
#pragma unroll
              for (int k = 1; k < 3; ++k) {
                sa = f2_add(sa, e2[k][0]);
                sb = f2_add(sb, e2[k][1]);
                sa = f2_add(sa, e2[k][2]);
                sb = f2_add(sb, e2[k][3]);
              }
              float slo, shi;
              f2_unpack(f2_add(sa, sb), slo, shi);
              const float lm = (slo + shi) * (1.0f / 24.0f);
              const uint64_t nlm = f2_pack(-lm, -lm);
              uint64_t qa = 0, qb = 0;
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                uint64_t d = f2_add(e2[k][0], nlm);
                qa = f2_fma(d, d, qa);
                d = f2_add(e2[k][1], nlm);
                qb = f2_fma(d, d, qb);
                d = f2_add(e2[k][2], nlm);
                qa = f2_fma(d, d, qa);
                d = f2_add(e2[k][3], nlm);
                qb = f2_fma(d, d, qb);
              }
              float qlo, qhi;
              f2_unpack(f2_add(qa, qb), qlo, qhi);
              const float q = qlo + qhi;
              if (l == 0) {
                pst = Chan{24u, lm, q};
              } else {
                const float wb = __fdividef(1.0f, (float)(l + 1));
                const float d = lm - pst.mean;
                pst.mean = fmaf(d, wb, pst.mean);
                pst.m2 = (pst.m2 + q) + (d * d) * (24.0f * (1.0f - wb));
                pst.n += 24u;
              }
            }
            st = chan_merge(st, pst);
          }
        } else {
        // the last, partial piece of a slice: leaves of LEAF units a lane
        // (units lane, lane + 32, ...), empty units left out
        for (int u0 = 0; u0 < nu; u0 += 32 * LEAF) {
          uint64_t e2[LEAF][4];
          int cnt = 0;
#pragma unroll
          for (int k = 0; k < LEAF; ++k) {
            const int u = u0 + lane + 32 * k;
            if (u < nu) {
              ring_unit2<In>(slot, u, e2[k]);
              cnt += 8;
            }
          }
          if (cnt == 0) continue;
          if constexpr (MODE == kModeSoftmax) {
            // the leaf's maximum, then its sum of e^(x - max), folded into
            // the lane's (max, sum)
            float cm = -INFINITY;
#pragma unroll
            for (int k = 0; k < LEAF; ++k) {
              if (u0 + lane + 32 * k < nu) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float lo, hi;
                  f2_unpack(e2[k][q], lo, hi);
                  cm = fmaxf(cm, fmaxf(lo, hi));
                }
              }
            }
            float ls = 0.0f;
            if (cm != -INFINITY) {
              const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
              const uint64_t nmb2 = f2_pack(-cm * kLog2e, -cm * kLog2e);
              uint64_t acc = 0;
#pragma unroll
              for (int k = 0; k < LEAF; ++k) {
                if (u0 + lane + 32 * k < nu) {
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    float lo, hi;
                    f2_unpack(f2_fma(e2[k][q], l2e2, nmb2), lo, hi);
                    acc = f2_add(acc, f2_pack(ex2_approx(lo), ex2_approx(hi)));
                  }
                }
              }
              float alo, ahi;
              f2_unpack(acc, alo, ahi);
              ls = alo + ahi;
            }
            ms_combine(m, sm, cm, ls);
          } else {
            // two-pass about the leaf's mean, two elements per instruction
            // (even and odd elements in the two halves)
            uint64_t sa = 0, sb = 0;
#pragma unroll
            for (int k = 0; k < LEAF; ++k) {
              if (u0 + lane + 32 * k < nu) {
                sa = f2_add(sa, e2[k][0]);
                sb = f2_add(sb, e2[k][1]);
                sa = f2_add(sa, e2[k][2]);
                sb = f2_add(sb, e2[k][3]);
              }
            }
            float slo, shi;
            f2_unpack(f2_add(sa, sb), slo, shi);
            const float lm = __fdividef(slo + shi, (float)cnt);
            const uint64_t nlm = f2_pack(-lm, -lm);
            uint64_t qa = 0, qb = 0;
#pragma unroll
            for (int k = 0; k < LEAF; ++k) {
              if (u0 + lane + 32 * k < nu) {
                uint64_t d = f2_add(e2[k][0], nlm);
                qa = f2_fma(d, d, qa);
                d = f2_add(e2[k][1], nlm);
                qb = f2_fma(d, d, qb);
                d = f2_add(e2[k][2], nlm);
                qa = f2_fma(d, d, qa);
                d = f2_add(e2[k][3], nlm);
                qb = f2_fma(d, d, qb);
              }
            }
            float qlo, qhi;
            f2_unpack(f2_add(qa, qb), qlo, qhi);
            st = chan_merge(st, Chan{(uint32_t)cnt, lm, qlo + qhi});
          }
        }
        }
        __syncwarp();
        if (lane == 0 && it + stages < total) issue(it + stages);
      }
      // ---- publish the warp's state for row j (slot wst[par] is free once
      // the reducer has finished row j - 2)
      if (j >= 2) wait(&rowres[par], ((uint32_t)(j - 2) >> 1) & 1u);
      if constexpr (MODE == kModeSoftmax) {
        ms_warp<32>(m, sm);
        if (lane == 0) {
          wst[par][warp][0] = __float_as_uint(m);
          wst[par][warp][1] = __float_as_uint(sm);
        }
      } else {
        st = chan_warp<32>(st);
        if (lane == 0) {
          wst[par][warp][0] = st.n;
          wst[par][warp][1] = __float_as_uint(st.mean);
          wst[par][warp][2] = __float_as_uint(st.m2);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rowbar[par]);
      if constexpr (NPASS == 2) {
        // ---- pass 2: the row's result, then this warp's pieces rewritten
        wait(&rowres[par], ph);
        const float r0 = res[par][0], r1 = res[par][1];
        for (int p = 0; p < np; ++p, ++it) {
          if ((int)(it % (uint32_t)NW) != warp) continue;
          const int s = (int)(it % stages);
          wait(&full[s], (it / stages) & 1u);
          const unsigned char *slot = ring + (size_t)s * piece;
          const int nu = piece_units(p);
          if constexpr (MODE == kModeSoftmax) {
            const float Mx = r0, inv = r1;
            const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
            const uint64_t nmb2 = f2_pack(-Mx * kLog2e, -Mx * kLog2e), inv2 = f2_pack(inv, inv);
            float *yp = y + row * cols + b0 + (int64_t)p * UPP * 8;
            for (int u = lane; u < nu; u += 32) {
              uint64_t e2[4];
              float o[8];
              ring_unit2<In>(slot, u, e2);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                float lo, hi;
                f2_unpack(f2_fma(e2[k], l2e2, nmb2), lo, hi);
                f2_unpack(f2_mul(f2_pack(ex2_approx(lo), ex2_approx(hi)), inv2), o[2 * k],
                          o[2 * k + 1]);
              }
              if (Mx == -INFINITY) {
#pragma unroll
                for (int k = 0; k < 8; ++k) o[k] = 0.0f;
              }
              st_stream_v8(yp + (int64_t)u * 8, o);
            }
          } else {
            const uint64_t mu2 = f2_pack(r0, r0), rs2 = f2_pack(r1, r1);
            const int64_t c0 = b0 + (int64_t)p * UPP * 8;
            const bool gb32 = aligned32(gamma + c0, beta + c0);
            uint16_t *yp = ybf + row * cols + c0;
            // 2 units a lane per round: every gamma / beta load of the round
            // (through L2) goes out before the first is used
            constexpr int RU = 2;
            for (int u0 = lane; u0 < nu; u0 += 32 * RU) {
              float g[RU][8], bt[RU][8];
#pragma unroll
              for (int k = 0; k < RU; ++k) {
                const int u = u0 + 32 * k;
                if (u < nu)
                  load_gamma_beta<8>(gamma + c0, beta + c0, (int64_t)u * 8, gb32, g[k], bt[k]);
              }
#pragma unroll
              for (int k = 0; k < RU; ++k) {
                const int u = u0 + 32 * k;
                if (u < nu) {
                  uint64_t e2[4];
                  ring_unit2<In>(slot, u, e2);
                  uint32_t pk[4];
#pragma unroll
                  for (int q = 0; q < 4; ++q) {
                    // fmaf((x - mu) * rs, gamma, beta), two elements at a time
                    const uint64_t t = f2_mul(f2_sub(e2[q], mu2), rs2);
                    float lo, hi;
                    f2_unpack(f2_fma(t, f2_pack(g[k][2 * q], g[k][2 * q + 1]),
                                     f2_pack(bt[k][2 * q], bt[k][2 * q + 1])), lo, hi);
                    pk[q] = bf16x2_bits(lo, hi);
                  }
                  *reinterpret_cast<uint4 *>(yp + (int64_t)u * 8) =
                      make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0 && it + stages < total) issue(it + stages);
        }
      }
    }
    // no copy may still be landing when the CTA exits, even if a wait above
    // gave up: wait (bounded, regardless of the timeout flag) for the last
    // copy into each of the warp's slots
    if (lane == 0) {
      for (uint32_t s0 = (uint32_t)warp; s0 < stages; s0 += NW) {
        if (s0 >= total) continue;
        const uint32_t lastk = s0 + ((total - 1 - s0) / stages) * stages;
        if (!mbar_wait_bounded(&full[s0], (lastk / stages) & 1u, kWaitBudget))
          set_error(err, kErrTimeout);
      }
    }
  }
  // no CTA leaves while a peer may still write its exchange slots
  if (C > 1) cluster_sync();
}

template <class In, int MODE>
int launch_mode(const void *x, int64_t rows, int64_t cols, float eps, float *y, float *mean,
                float *rstd, const float *gamma, const float *beta, uint16_t *ybf, int C,
                bool shrink, int *C_out, cudaStream_t s, const DevInfo &d) {
  auto kern = k_rowwise_ring<In, MODE>;
  constexpr int64_t E = (int64_t)sizeof(typename In::S);
  if (C < 1 || C > 16 || cols % 8 != 0) return RR_ERR_INVALID;
  // one CTA per SM (the ring alone holds more than half the SM's shared
  // memory) when every cluster gets its own SMs, else two
  const bool one_per_sm = rows * C <= d.sm_count;
  const uint32_t piece = one_per_sm ? kRingPieceBig : kRingPieceSmall;
  const size_t smem = (size_t)kRingStages * piece;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(kRingStages * kRingPieceBig));
  if (e != cudaSuccess) return cuda_status(e);
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_status(e);
  }
  // a few rows: the largest C (down to 2) whose clusters all run at once
  int active = occupancy_clusters((const void *)kern, kRingThreads, smem, C, d.device);
  while (shrink && one_per_sm && C > 2 && active < rows) {
    --C;
    active = occupancy_clusters((const void *)kern, kRingThreads, smem, C, d.device);
  }
  if (active < 1) return RR_ERR_UNSUPPORTED;
  const int64_t chunk = ((cols + C - 1) / C + 7) & ~int64_t(7);
  if (chunk * E > (int64_t)0xffffffffLL) return RR_ERR_INVALID;
  int64_t ncl = rows < active ? rows : active;
  if (ncl < 1) ncl = 1;
  // a CTA's items (pieces of all its rows and passes) are counted in 32 bits
  if (((rows + ncl - 1) / ncl) * 2 * ((chunk * E) / piece + 1) > 0x7fffffffLL) return RR_ERR_INVALID;
  if (ncl * C > 0x7fffffffLL) return RR_ERR_INVALID;
  *C_out = C;
  if (log_enabled())
    std::fprintf(stderr, "rr: %s ring rows=%lld cols=%lld C=%d clusters=%lld (active %d) piece=%u\n",
                 MODE == kModeSoftmax ? "softmax" : (MODE == kModeStats ? "lnstats" : "layernorm"),
                 (long long)rows, (long long)cols, C, (long long)ncl, active, piece);
  return cuda_status(launch_kernel(kern, dim3((unsigned)(ncl * C)), dim3(kRingThreads), smem, s, C,
                                   (const typename In::S *)x, rows, cols, chunk, piece, eps, y,
                                   mean, rstd, gamma, beta, ybf, d.err_word));
}

}  // namespace

int launch_rowwise_ring(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                        float eps, float *y, float *mean, float *rstd, const float *gamma,
                        const float *beta, uint16_t *ybf, int C, bool shrink, int *C_out,
                        cudaStream_t s, const DevInfo &d) {
  if (in_dtype == RR_BF16) {
    switch (mode) {
      case kModeSoftmax: return launch_mode<InBF16, kModeSoftmax>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
      case kModeStats: return launch_mode<InBF16, kModeStats>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
      default: return launch_mode<InBF16, kModeLayernorm>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
    }
  }
  switch (mode) {
    case kModeSoftmax: return launch_mode<InF32, kModeSoftmax>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
    case kModeStats: return launch_mode<InF32, kModeStats>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
    default: return launch_mode<InF32, kModeLayernorm>(x, rows, cols, eps, y, mean, rstd, gamma, beta, ybf, C, shrink, C_out, s, d);
  }
}

}  // namespace rr
