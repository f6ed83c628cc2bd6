// rr_device.cuh -- device primitives for sm_103a shared by the librr kernels:
// monoid ops, 128/256-bit streaming loads, warp and block trees, the cluster
// all-reduce over distributed shared memory, and bounded mbarrier waits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rr {

// Status bits OR-ed into the per-device error word by kernels.
constexpr int kErrTimeout = 1;

// ---------------------------------------------------------------------------
// Monoids.  The "reduce" page (algorithm/gpu/rowwise) folds tiles into a
// monoid state; the "cluster_allreduce" page names add, max and min as the
// associative combine functions on 32-bit types.
//
// max / min on fp32 are made independent of the fold order down to the bits:
// max(+0,-0) = +0 and min(+0,-0) = -0 in either order, and a NaN operand
// makes the result NaN (canonicalised to 0x7fc00000 by finalize()).  The
// PTX max.NaN / min.NaN instructions have exactly these semantics on
// sm_103a (checked on the device for every pair of +-0, +-1, +-inf and
// NaNs, and by the signed-zero / NaN GPU tests), so each fold step is one
// instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float min_nan(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

struct SumF32 {
  using T = float;
  static __device__ __forceinline__ T id() { return 0.0f; }
  static __device__ __forceinline__ T f(T a, T b) { return __fadd_rn(a, b); }
  static __device__ __forceinline__ T finalize(T a) { return a; }
};

struct MaxF32 {
  using T = float;
  static __device__ __forceinline__ T id() { return __int_as_float(0xff800000); }
  static __device__ __forceinline__ T f(T a, T b) { return max_nan(a, b); }
  static __device__ __forceinline__ T finalize(T a) {
    return (a != a) ? __int_as_float(0x7fc00000) : a;
  }
};

struct MinF32 {
  using T = float;
  static __device__ __forceinline__ T id() { return __int_as_float(0x7f800000); }
  static __device__ __forceinline__ T f(T a, T b) { return min_nan(a, b); }
  static __device__ __forceinline__ T finalize(T a) {
    return (a != a) ? __int_as_float(0x7fc00000) : a;
  }
};

struct SumI32 {
  using T = int;
  static __device__ __forceinline__ T id() { return 0; }
  static __device__ __forceinline__ T f(T a, T b) {
    return (int)((unsigned)a + (unsigned)b);  // wraps modulo 2^32
  }
  static __device__ __forceinline__ T finalize(T a) { return a; }
};

struct MaxI32 {
  using T = int;
  static __device__ __forceinline__ T id() { return (int)0x80000000; }
  static __device__ __forceinline__ T f(T a, T b) { return a > b ? a : b; }
  static __device__ __forceinline__ T finalize(T a) { return a; }
};

struct MinI32 {
  using T = int;
  static __device__ __forceinline__ T id() { return 0x7fffffff; }
  static __device__ __forceinline__ T f(T a, T b) { return a < b ? a : b; }
  static __device__ __forceinline__ T finalize(T a) { return a; }
};

// 4-wide vector of the op's element type.
template <class T> struct Vec4;
template <> struct Vec4<float> { using type = float4; };
template <> struct Vec4<int> { using type = int4; };

// ---------------------------------------------------------------------------
// Streaming global loads: read-only path, no L1 allocation (each byte is
// used once).  16-byte and 32-byte (sm_100+ 256-bit) forms.  The asm is
// volatile so that a batch of loads written back to back is issued back to
// back (the compiler may not sink a load down to its first use), which keeps
// that many bytes in flight per thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_stream(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ int4 ld_stream(const int4 *p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// L2 eviction policies for loads (createpolicy): evict_last keeps lines a
// later kernel reads again ahead of other traffic; evict_first lets lines
// read for the last time go first.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// ld_stream_u4 with an L2 eviction policy.
__device__ __forceinline__ uint4 ld_stream_u4_hint(const void *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}
// 32 contiguous bytes (8 x 32-bit) in one instruction; p 32-byte aligned.
__device__ __forceinline__ void ld_stream_v8(const void *p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "l"(p));
}
// 32-byte streaming store (evict-first), p 32-byte aligned.
__device__ __forceinline__ void st_stream_v8(void *p, const float (&v)[8]) {
  asm volatile(
      "st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
      "f"(v[6]), "f"(v[7])
      : "memory");
}
__device__ __forceinline__ void st_stream_v4(void *p, float a, float b,
                                             float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <class Op, class V>
__device__ __forceinline__ typename Op::T fold4(typename Op::T acc, const V &v) {
  acc = Op::f(acc, v.x);
  acc = Op::f(acc, v.y);
  acc = Op::f(acc, v.z);
  acc = Op::f(acc, v.w);
  return acc;
}

// ---------------------------------------------------------------------------
// Warp and block trees (fixed shape, so the combine order is fixed).
// ---------------------------------------------------------------------------
template <class T> __device__ __forceinline__ T shfl_xor(T v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}

// Butterfly over aligned segments of SEG lanes; every lane of a segment ends
// with the segment's result.
template <class Op, int SEG>
__device__ __forceinline__ typename Op::T warp_allreduce(typename Op::T v) {
#pragma unroll
  for (int o = SEG / 2; o > 0; o >>= 1) v = Op::f(v, shfl_xor(v, o));
  return v;
}

__host__ __device__ constexpr int pow2_ceil(int n) { return n <= 1 ? 1 : 2 * pow2_ceil((n + 1) / 2); }

// Block reduce: warp trees, then warp 0 folds the per-warp values.  The
// result is valid in thread 0.  `red` holds THREADS/32 elements; the caller
// must __syncthreads() before reusing it.
template <class Op, int THREADS>
__device__ __forceinline__ typename Op::T block_reduce(typename Op::T v,
                                                       typename Op::T *red) {
  constexpr int NW = THREADS / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_allreduce<Op, 32>(v);
  if (NW == 1) return v;
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = (lane < NW) ? red[lane] : Op::id();
    v = warp_allreduce<Op, pow2_ceil(NW)>(v);
  }
  return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  First statement of every kernel: wait until
// the previous grid in the stream has completed and its memory operations are
// visible (griddepcontrol.wait).  The launch attribute lets this grid be set
// up while the previous one drains; the dependency on the previous grid is
// released as its blocks exit (no explicit launch_dependents: releasing it at
// a kernel's start let the next grid's CTAs take SM slots from persistent
// cluster kernels and slowed them).  Without the attribute the wait does
// nothing.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_begin() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next grid launch once every CTA of this one has called it or
// exited, for a kernel one wave deep whose CTAs have issued their last
// loads; the next grid's pdl_begin still waits for this grid to complete.
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block cluster primitives (PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nid_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Cluster-wide execution barrier; arrive orders this thread's earlier memory
// operations (release), wait makes the peers' earlier ones visible (acquire).
// Every thread of every CTA of the cluster must call it; the non-.aligned
// form does not require the warp to be converged.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\t"
               "barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  return __uint_as_float(ld_dsmem_u32(addr));
}
// 16 bytes into the shared memory of a peer CTA (addr from map_peer, 16-byte
// aligned); ordered before a later release-arrive of the same thread.
__device__ __forceinline__ void st_dsmem_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

template <class T> __device__ __forceinline__ uint32_t to_bits(T v);
template <> __device__ __forceinline__ uint32_t to_bits<float>(float v) { return __float_as_uint(v); }
template <> __device__ __forceinline__ uint32_t to_bits<int>(int v) { return (uint32_t)v; }
template <class T> __device__ __forceinline__ T from_bits(uint32_t u);
template <> __device__ __forceinline__ float from_bits<float>(uint32_t u) { return __uint_as_float(u); }
template <> __device__ __forceinline__ int from_bits<int>(uint32_t u) { return (int)u; }

// ---------------------------------------------------------------------------
// cluster_allreduce ("cluster_allreduce" page).
//
// `slot` is a __shared__ array of 2*W elements declared at the same place in
// every CTA of the cluster (a static __shared__ array of the kernel, never an
// offset computed at run time), so mapa finds the peers' copies.  `vals` is
// this CTA's block-reduced vector, valid in thread 0.  Thread 0 publishes it
// in slot[0:W]; after a cluster barrier it reads slot[0:W] of every rank
// 0..C-1 and folds them in rank order; it writes the result to slot[W:2W],
// from where every thread of the block picks it up.  Because every CTA folds
// the same values in the same order, every CTA gets the same bits.
//
// tail_sync = true ends with a second cluster barrier: once it passes, no
// peer will read this slot again, so the next combine may reuse it.
// tail_sync = false skips that barrier ("cluster_allreduce" page, the
// need_tail_sync parameter) and the caller alternates two slots, A, B, A, ...
// Why that is safe: combine k+1 writes slot B, which no peer reads during
// combine k; and before any CTA writes slot A again in combine k+2 it has
// passed the barrier of combine k+1, which every peer reaches only after
// finishing its reads of slot A in combine k.  So the lead of the fastest CTA
// over the slowest is bounded by one combine.  The kernel must still end
// with cluster_sync(), so that no CTA exits (and its shared memory goes away)
// while a peer may still read its last slot.  With C == 1 no barrier is
// needed: the call only publishes thread 0's values to the block.
// ---------------------------------------------------------------------------
template <class Op, int W>
__device__ __forceinline__ void cluster_allreduce(typename Op::T *slot,
                                                  const typename Op::T (&vals)[W],
                                                  uint32_t C, bool tail_sync,
                                                  typename Op::T (&out)[W]) {
  using T = typename Op::T;
  if (C > 1) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int j = 0; j < W; ++j) slot[j] = vals[j];
    }
    cluster_sync();
    if (threadIdx.x == 0) {
      // all C loads of an element go out before the first is folded (C <= 16),
      // so the gather costs about one distributed-shared-memory round trip
      const uint32_t base = smem_u32(slot);
#pragma unroll
      for (int j = 0; j < W; ++j) {
        uint32_t raw[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if ((uint32_t)r < C) raw[r] = ld_dsmem_u32(map_peer(base + 4u * j, (uint32_t)r));
        T acc = from_bits<T>(raw[0]);
#pragma unroll
        for (int r = 1; r < 16; ++r)
          if ((uint32_t)r < C) acc = Op::f(acc, from_bits<T>(raw[r]));
        slot[W + j] = acc;
      }
    }
  } else {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int j = 0; j < W; ++j) slot[W + j] = vals[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < W; ++j) out[j] = slot[W + j];
  if (C > 1 && tail_sync) cluster_sync();
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (the copy engine writes the CTA's own shared
// memory; no multicast).  Every wait is bounded: after `budget` polls it
// gives up and returns false, and the caller records kErrTimeout.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Raise the expected transaction count of the current phase without
// arriving (the arrival comes later, e.g. after plain stores it must
// release).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  int64_t budget) {
  for (int64_t i = 0; i < budget; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Bulk copy global -> this CTA's shared memory; bytes % 16 == 0, both
// addresses 16-byte aligned.  Completion is signalled on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Arrive (release, cluster scope) on the mbarrier at `bar`'s offset in the
// shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *bar, uint32_t rank) {
  const uint32_t a = map_peer(smem_u32(bar), rank);
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a)
               : "memory");
}
// Relaxed remote arrive that also raises the expected transaction count of
// the peer's mbarrier by `bytes` (the bytes a bulk copy will deliver there).
__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint64_t *bar, uint32_t rank,
                                                             uint32_t bytes) {
  const uint32_t a = map_peer(smem_u32(bar), rank);
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(a),
               "r"(bytes)
               : "memory");
}
// Bulk copy from this CTA's shared memory into the shared memory of CTA
// `rank` of the cluster (same offsets as `dst_local` / `bar_local` here);
// completion is counted on that CTA's mbarrier.  bytes % 16 == 0.
__device__ __forceinline__ void bulk_s2peer(void *dst_local, const void *src, uint32_t bytes,
                                            uint64_t *bar_local, uint32_t rank) {
  const uint32_t d = map_peer(smem_u32(dst_local), rank);
  const uint32_t b = map_peer(smem_u32(bar_local), rank);
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(d),
      "r"(smem_u32(src)), "r"(bytes), "r"(b)
      : "memory");
}
// Relaxed remote arrive: orders nothing, only counts.  For signals whose
// payload is already guaranteed by data dependences (e.g. "my loads of your
// buffer have returned").
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint64_t *bar, uint32_t rank) {
  const uint32_t a = map_peer(smem_u32(bar), rank);
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(a)
               : "memory");
}
// Wait (acquire, cluster scope) for phase `parity` of a local mbarrier whose
// arrivals come from peer CTAs.
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded waits that give up at once after the CTA's first timeout (`dead`,
// a shared flag), so that a broken protocol costs one budget, not one per
// wait.
__device__ __forceinline__ bool mbar_wait_or_die(uint64_t *bar, uint32_t parity, int64_t budget,
                                                 volatile int *dead, bool cluster_scope) {
  for (int64_t i = 0; i < budget; ++i) {
    if (cluster_scope ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity))
      return true;
    if (*dead) return false;
  }
  *dead = 1;
  return false;
}
// Barrier over the first `n` threads of the CTA (named barrier `id`, 1..15).
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void set_error(int *err, int code) {
  if (err) atomicOr(err, code);
}

// Polls of a bounded mbarrier wait before it gives up.  Each poll is a
// try_wait that may itself suspend for a short, hardware-defined time, so
// the budget is of the order of a second.
constexpr int64_t kWaitBudget = int64_t(1) << 20;

}  // namespace rr
