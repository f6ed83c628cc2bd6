// rr_internal.h -- host-side interface between the C-ABI layer (api.cu) and
// the per-family launchers (reduce.cu, rowwise.cu, combine.cu, cluster.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rr {

struct DevInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;     // bytes of shared memory a CTA may opt into
  int cluster_launch = 0;     // device supports cluster launch
  int *err_word = nullptr;    // device error word (4 bytes), zeroed
};

// Returns the cached info of the current device (creating the error word on
// first use), or nullptr with *status set on failure.
const DevInfo *current_device(int *status);

// ---- reduce (reduce.cu)
// Largest cluster size in {16, 8, 4, 2, 1} <= `want` that the split-K kernel
// for (op, dtype) can co-schedule on this device (0 if not even 1).
int splitk_max_cluster(int op, int dtype, int want, const DevInfo &d);
int launch_reduce(const void *x, int64_t rows, int64_t cols, int op, int dtype,
                  void *out, cudaStream_t s, int tier, int C, int ewt,
                  void *rank_out, const DevInfo &d);

// Multi-cluster split-K (G clusters of C CTAs per row, partials in ws).
int launch_reduce_splitk_multi(const void *x, int64_t rows, int64_t cols, int op, int dtype,
                               void *out, int C, int G, void *ws, cudaStream_t s);

// ---- reduction over a non-last axis (axis.cu)
// Largest cluster size in {16, 8, 4, 2} <= want the split-K axis kernel can
// co-schedule, else 1.
int axis_max_cluster(int want, const DevInfo &d);
// One resolved launch of rr_reduce_axis for inner > 1.
struct AxisPlan {
  int tier = 0;  // RR_TIER_TILED, RR_TIER_WARP, RR_TIER_BLOCK or RR_TIER_SPLITK
  int C = 1;     // split-K cluster size
  int E = 1;     // tiled: rows per thread (1, 2 or 4)
  int V = 1;     // warp / block / split-K: 4 (16-byte loads; inner % 4 == 0
                 // and x 16-byte aligned) or 1
  int lg_L = 0;  // warp / block / split-K: log2 of lanes per axis position
                 // (tile = (1 << lg_L) * V adjacent rows)
  int G = 1;     // block / split-K: independent CTAs / clusters per tile; G > 1
                 // writes G partials per output to the workspace, then folds
  bool slab = false;  // a warp (warp tier) or a CTA (block tier) per contiguous slab
                      // x[o, :, :] (inner 2, 3, 5, 6 or 7)
};
int launch_reduce_axis(const void *x, int64_t outer, int64_t axis, int64_t inner, int op,
                       int dtype, void *out, const AxisPlan &plan, void *workspace,
                       cudaStream_t s, const DevInfo &d);

// ---- softmax / layernorm statistics (rowwise.cu)
// The caller's workspace for the grid form (rowgrid.cu): `ws` (16-byte
// aligned, or null: no grid form) of `bytes` bytes; `splits` > 0 forces
// the grid form with that many CTAs per row.
struct RowWs {
  void *ws = nullptr;
  size_t bytes = 0;
  int splits = 0;
};
// tier: RR_TIER_AUTO, RR_TIER_WARP, RR_TIER_BLOCK or RR_TIER_SPLITK; C:
// split-K cluster size, or the warp tier's lanes per row (0 = automatic).
// *tier_out receives tier | (width & 0xff) << 8 | staged << 16 | ring << 17
// | grid << 18 | (width >> 8) << 19 (width: lanes per row for the warp
// tier, CTAs per row for the grid form, else the cluster size).
int launch_softmax(const void *x, int64_t rows, int64_t cols, int in_dtype,
                   float *out, cudaStream_t s, const DevInfo &d, int *tier_out,
                   int tier, int C, const RowWs &w);
int launch_layernorm_stats(const void *x, int64_t rows, int64_t cols,
                           int in_dtype, float eps, float *mean, float *rstd,
                           cudaStream_t s, const DevInfo &d, int *tier_out,
                           int tier, int C, const RowWs &w);

// Layernorm (statistics + rewrite, bf16 out); mean / rstd may be null.
int launch_layernorm(const void *x, int64_t rows, int64_t cols, int in_dtype, float eps,
                     const float *gamma, const float *beta, uint16_t *y, float *mean,
                     float *rstd, cudaStream_t s, const DevInfo &d, int *tier_out, int tier,
                     int C, const RowWs &w);

// ---- tier choice of the row operations (rowwise.cu, host only)
// Rows per SM from which the automatic choice takes the warp tier for rows
// that fit it; below that a CTA per row finishes sooner.  The layernorm
// rewrite, whose lanes also load gamma and beta for every vector they
// write, needs more rows to come out ahead.
constexpr int kRowWarpMinRowsPerSM = 4;
constexpr int kRowWarpMinRowsPerSMRewrite = 8;
// tier RR_TIER_WARP (width = lanes per row), RR_TIER_SPLITK (width =
// cluster size) or RR_TIER_BLOCK (width 1); tier < 0 when a forced choice
// cannot run.  `staged`: the block / split-K tier with the row's slices
// staged in shared memory (rowstaged.cu).
struct RowPlan {
  int tier;
  int width;
  bool staged;
  bool ring = false;  // streamed through a shared-memory ring (rowring.cu)
  bool half = false;  // block tier, row in registers read as 8-byte vectors
  bool grid = false;  // split-K over a plain grid, width CTAs per row (rowgrid.cu)
  bool chunk = false; // block tier, statistics of a row not 16-byte aligned as head + vectors + tail
  bool twopass = false;  // rewrite of many long rows: ring statistics, then launch_ln_apply
};
// Forced (tier, C) or automatic choice for rows x cols of `in_dtype`; `vec`:
// cols is a multiple of the 16-byte vector and every operand meets the
// register forms' alignment; `mode`: 0 softmax, 1 layernorm statistics, 2
// layernorm rewrite.  A forced split-K cluster larger than max_cluster
// cannot run.
// out_vec: for rows that are not aligned vectors, whether the output shares
// x's offset within a 16-byte chunk (true for 16-byte aligned bases).
// half: the rows are not 16-byte aligned vectors but every operand allows the
// 8-byte vector register form (cols a multiple of 4 bf16 / 2 fp32, x and the
// outputs 8-byte aligned, gamma / beta as that form loads them).
// grid_ok: a workspace is at hand and the operands meet the grid form's
// alignment (as the ring form's).
RowPlan plan_rowwise(int64_t rows, int64_t cols, int in_dtype, bool vec, int mode, int tier,
                     int C, int sm_count, int max_cluster, bool out_vec = true, bool half = false,
                     bool grid_ok = false);
// Vectors per row up to which the block tier holds the row in registers
// (256 threads x 8 vectors).
constexpr int64_t kRowRegMaxVec = 2048;

// ---- staged row operations (rowstaged.cu)
// Largest slice a CTA stages in shared memory: two such CTAs fit on an SM.
#ifndef RR_STAGE_MAX_KB
#define RR_STAGE_MAX_KB 96
#endif
constexpr int64_t kStageMaxBytes = RR_STAGE_MAX_KB * 1024;
// Elements per CTA slice for a cluster of C (a multiple of 8); -1 if C < 1.
int64_t rowwise_staged_chunk(int64_t cols, int C);
// Smallest cluster size (a power of two up to min(16, max_cluster)) whose
// slices fit kStageMaxBytes (rows that are not 16-byte aligned stage up to
// 8 elements more per slice); 0 if none does.
int rowwise_staged_cluster(int64_t cols, int in_dtype, int max_cluster, bool aligned = true);
// mode as launch_rowwise_warp.  `aligned`: every operand meets the vector
// forms' alignment (as for the warp tier); otherwise the misaligned form
// runs, for any element-aligned x and outputs.
int launch_rowwise_staged(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                          float eps, float *y, float *mean, float *rstd, const float *gamma,
                          const float *beta, uint16_t *ybf, int C, bool aligned, cudaStream_t s,
                          const DevInfo &d);

// ---- streamed row operations (rowring.cu)
// Rows whose second pass (softmax, layernorm rewrite) re-reads them from L2:
// the ring form takes them while the rows in flight hold at most this many
// bytes.
constexpr int64_t kRingL2Bytes = int64_t(64) << 20;
// mode as launch_rowwise_warp; x 16-byte aligned, cols a multiple of 8, y
// 32-byte aligned (softmax), ybf / gamma / beta 16-byte aligned (rewrite).
// C: cluster size (1..16, any value); with `shrink` a C whose clusters
// cannot all run at once is lowered (to 2 at least) until they can.  *C_out
// receives the cluster size launched.
int launch_rowwise_ring(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                        float eps, float *y, float *mean, float *rstd, const float *gamma,
                        const float *beta, uint16_t *ybf, int C, bool shrink, int *C_out,
                        cudaStream_t s, const DevInfo &d);
// ---- grid form of the row operations (rowgrid.cu)
// Slices of at least kRowGridMinSlice elements, at most kRowGridMaxSplits
// CTAs per row.
constexpr int64_t kRowGridMinSlice = 2048;
constexpr int kRowGridMaxSplits = 1024;
// CTAs per row for rows x cols: about 4 CTAs per SM over all rows.
int rowgrid_splits(int64_t rows, int64_t cols, int sm_count);
// Workspace bytes of the grid form: a 16-byte state per CTA.
inline size_t rowgrid_ws_bytes(int64_t rows, int G) { return (size_t)rows * (size_t)G * 16; }
// mode as launch_rowwise_warp; x 16-byte aligned, cols a multiple of 8, y
// 32-byte aligned (softmax), ybf / gamma / beta 16-byte aligned (rewrite),
// ws 16-byte aligned with at least rowgrid_ws_bytes(rows, G) bytes, not
// overlapping any operand; RR_ERR_INVALID otherwise.  Two launches.
int launch_rowgrid(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols, float eps,
                   float *y, float *mean, float *rstd, const float *gamma, const float *beta,
                   uint16_t *ybf, int G, void *ws, size_t ws_bytes, cudaStream_t s,
                   const DevInfo &d);
// The layernorm rewrite of rows whose (mean, rstd) are already in mean_in /
// rstd_in: x read again, y = (x - mean) rstd gamma + beta in bf16, gamma /
// beta loaded once per column block of a group of rows.  x 16-byte aligned,
// cols a multiple of 8, ybf / gamma / beta 16-byte aligned; RR_ERR_INVALID
// otherwise.  One launch.
int launch_ln_apply(int in_dtype, const void *x, int64_t rows, int64_t cols, const float *mean_in,
                    const float *rstd_in, const float *gamma, const float *beta, uint16_t *ybf,
                    cudaStream_t s, const DevInfo &d);
// Rows from which rr_layernorm, given a workspace, takes the two-pass form
// when there are at least as many rows as SMs (bytes of x a row).
constexpr int64_t kRowTwoPassMinBytes = 256 << 10;
// Workspace bytes of the two-pass form: a row's mean and rstd.
inline size_t rowtwopass_ws_bytes(int64_t rows) { return (size_t)rows * 8; }
// ---- warp tier of the row operations (rowwarp.cu)
// A segment of L lanes per row holding NV 16-byte vectors per lane, NV a
// power of two up to kRowWarpMaxNV.
constexpr int kRowWarpMaxNV = 8;
constexpr int kRowWarpTargetNV = 4;  // automatic L: about this many vectors per lane
// Lanes per row for a row of nvec 16-byte vectors: `lanes` (1..32, a power
// of two) if it can hold the row, else 0; lanes == 0 picks one (for the
// layernorm rewrite when `rewrite`).  0 when the row does not fit the tier.
int rowwise_warp_lanes(int64_t nvec, int lanes, bool rewrite);
// Vectors per lane for nvec vectors over `lanes` lanes (a power of two).
int rowwise_warp_nv(int64_t nvec, int lanes);
// Warp tier for rows that are not aligned 16-byte vectors: a chunked form
// (the aligned 16-byte chunks covering the row, spread over the lanes as in
// the vector form) and, for the narrowest rows, an element-wise form of up
// to 32 * kRowWarpMaxElPerLane elements.
constexpr int kRowWarpMaxElPerLane = 32;
// Lanes per row of that tier: `lanes` if it can hold the row (a power of
// two), lanes == 0 picks one; 0 when the row does not fit.  out_vec: the
// output shares x's offset within a 16-byte chunk (rowwise_warp_out_vec).
int rowwise_warp_mis_lanes(int64_t cols, int in_dtype, int mode, bool out_vec, int lanes);
bool rowwise_warp_out_vec(int mode, int in_dtype, const void *x, const void *out);
int launch_rowwise_warp_mis(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                            float eps, float *y, float *mean, float *rstd, const float *gamma,
                            const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                            const DevInfo &d);
// The element-wise form alone (lanes and launch).
int rowwise_warp_el_lanes(int64_t cols, int lanes);
int launch_rowwise_warp_el(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                           float eps, float *y, float *mean, float *rstd, const float *gamma,
                           const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                           const DevInfo &d);
// mode 0 softmax (y), 1 statistics (mean, rstd), 2 layernorm (ybf; mean /
// rstd optional).  The caller has checked the alignment: cols a multiple
// of the 16-byte vector, x 16-byte aligned, y as the block tier's register
// form needs it, gamma / beta 16-byte aligned.
int launch_rowwise_warp(int mode, int in_dtype, const void *x, int64_t rows, int64_t cols,
                        float eps, float *y, float *mean, float *rstd, const float *gamma,
                        const float *beta, uint16_t *ybf, int lanes, cudaStream_t s,
                        const DevInfo &d);

// ---- split-K combine (combine.cu)
int launch_combine(const float *O, const float *m, const float *l, int P,
                   int64_t rows, int D, float scale_log2e, uint16_t *out,
                   cudaStream_t s, const DevInfo &d, int mode);

// ---- cluster all-reduce primitive (cluster.cu)
int launch_cluster_allreduce(const void *vals, int clusters, int C, int width,
                             int op, int dtype, int iters, int two_slot,
                             int64_t skew_cycles, void *res,
                             int64_t *mismatches, cudaStream_t s,
                             const DevInfo &d);
int launch_fill_selftest_values(void *vals, int64_t n, int dtype,
                                uint64_t seed, cudaStream_t s);
int launch_wait_timeout_probe(int64_t budget, cudaStream_t s, const DevInfo &d);

// Maps a CUDA error to an rr_status.
int cuda_status(cudaError_t e);

// Resident CTAs per SM of `func` with `threads` threads and `smem` bytes of
// dynamic shared memory on `device`, cached (the occupancy query costs
// microseconds per launch otherwise).  At least 1.
int occupancy_blocks(const void *func, int threads, size_t smem, int device);

// Largest number of co-resident clusters of `cluster` CTAs of `func`
// (cudaOccupancyMaxActiveClusters), cached; 0 if none can run or if
// `cluster` exceeds cluster_cap().  Every cluster launch of the library is
// checked through here.
int occupancy_clusters(const void *func, int threads, size_t smem, int cluster, int device);

// Largest cluster size the library launches: the environment variable
// RR_MAX_CLUSTER (1..16) read once, else 16.  Lets a process that shares
// the GPU keep clusters small; the automatic plans stay within it and a
// forced larger size returns RR_ERR_UNSUPPORTED.
int cluster_cap();

// Programmatic dependent launch: unless the environment variable RR_PDL is
// "0", every launch carries the programmatic-stream-serialization attribute,
// so a kernel is set up while the previous one in the stream drains.  Every
// kernel starts with pdl_begin() (rr_device.cuh), which waits for the
// previous grid to complete and its memory to be visible before touching
// global memory, so stream order is kept.
bool pdl_enabled();

// Launches `kern` on `s` with the programmatic-dependent-launch attribute
// (pdl_enabled()).  cluster == 0: a plain launch; cluster >= 1: a cluster
// launch with 1-D clusters of `cluster` CTAs -- a kernel that uses cluster
// instructions (distributed shared memory, bulk copies to shared::cluster,
// cluster barriers) must be launched this way even when the size is 1.
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cluster >= 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// True when the environment variable RR_LOG is set to a non-zero value:
// launchers then print their tier and launch configuration to stderr.
bool log_enabled();

}  // namespace rr
