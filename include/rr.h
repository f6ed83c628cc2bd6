/*
 * rr.h -- C ABI of librr.so: deterministic row-wise monoid reductions on
 * NVIDIA GB300 (sm_103a), the cluster all-reduce they are built on, and the
 * split-K attention-output combine.
 *
 * Sources (Mojo API documentation pages; cited by title and section):
 *   [CA] "cluster_allreduce" (max/gpu/primitives/cluster): description,
 *        parameters combine_fn / cluster_size / need_tail_sync, arg slot.
 *   [RW] "reduce" (algorithm/gpu/rowwise): tier semantics (warp, block,
 *        tiled, serial, split-K), the stateless and the state-carrying
 *        overloads, pjoin.
 *   [FA] "fa4_splitk_reduce_scatter_write" (kernels/nn/attention/gpu/nvidia/
 *        sm100/softmax_warp): split-K pass 2, band per partition, stage,
 *        publish, combine, bf16 store, terminal cluster sync.
 *
 * Conventions for every entry point
 *   - Pointers named x, out, O, m, l, mean, rstd, vals, res are DEVICE
 *     pointers owned by the caller; tensors are dense row-major (C order).
 *     The library never frees or retains them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work and return, unless stated otherwise.
 *   - Return value: an rr_status.  Arguments are validated on the host
 *     before anything is enqueued; an invalid call enqueues nothing.  No
 *     exception crosses this ABI.
 *   - rows == 0 is a no-op returning RR_OK.
 *   - The library allocates only a 4-byte device error word per device
 *     (on first use) and caches device properties; rr_cluster_allreduce_
 *     selftest also allocates and frees its own scratch.
 *   - Results are deterministic: the same inputs, shapes, pointer
 *     alignments and options give the same bits on every run (no float
 *     atomics, no occupancy-dependent partitioning of a row).
 *   - Launches carry the programmatic-dependent-launch attribute (the
 *     environment variable RR_PDL=0 turns it off): a kernel is set up
 *     while the previous one in the stream drains, and waits for it to
 *     complete before touching memory, so stream order is kept.
 *   - Cluster sizes: the library launches clusters of at most 16 CTAs and
 *     at most RR_MAX_CLUSTER (environment variable, 1..16, read once) when
 *     that is set; automatic plans stay within it, and a forced larger
 *     cluster size returns RR_ERR_UNSUPPORTED.
 */
#ifndef RR_H_
#define RR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RR_OK = 0,
    RR_ERR_INVALID = 1,     /* bad argument: null pointer, negative size,
                               unsupported (op, dtype), bad P / D, aliasing */
    RR_ERR_UNSUPPORTED = 2, /* valid request the device cannot run, e.g. no
                               active cluster of the requested size */
    RR_ERR_CUDA = 3,        /* a CUDA runtime call failed */
    RR_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
    RR_ERR_MISMATCH = 5     /* a self-test found a result that differs */
} rr_status;

typedef enum { RR_OP_SUM = 0, RR_OP_MAX = 1, RR_OP_MIN = 2 } rr_op;

typedef enum { RR_F32 = 0, RR_I32 = 1, RR_BF16 = 2 } rr_dtype;

/* Reduction tiers of [RW] "tier semantics". */
typedef enum {
    RR_TIER_AUTO = 0,
    RR_TIER_WARP = 1,    /* a warp segment per row: lane i takes element i
                            for rows of up to 32, and lanes stride longer
                            rows */
    RR_TIER_TILED = 2,   /* a thread owns emit_tile_width adjacent rows; no
                            cross-thread combine ([RW] tiled and serial tiers:
                            emit_tile_width 1 is the serial tier) */
    RR_TIER_BLOCK = 3,   /* a CTA per row, threads stride the axis */
    RR_TIER_SPLITK = 4   /* a cluster of C CTAs per row, combined through
                            distributed shared memory ([CA]) */
} rr_tier;

/*
 * Options of rr_reduce_ex.  Zero-initialise and set what you need.
 *   tier            RR_TIER_AUTO or a forced tier.
 *   cluster_size    split-K: 0 = automatic, else 1, 2, 4, 8 or 16.
 *   two_slot        reserved for multi-combine kernels (ignored by reduce,
 *                   which combines once per row).
 *   emit_tile_width tiled tier: rows per thread, 0 = automatic, else 1, 2, 4.
 *   rank_out        split-K only, optional device pointer to rows * C
 *                   elements of the output type: rank r of the cluster of
 *                   row i writes its copy of the combined result to
 *                   rank_out[i * C + r].  Every copy is bit-identical ([CA]
 *                   description); this exposes it for checking.
 */
typedef struct {
    int tier;
    int cluster_size;
    int two_slot;
    int emit_tile_width;
    void *rank_out;
} rr_reduce_opts;

/*
 * rr_reduce -- out[i] = x[i,0] (+) x[i,1] (+) ... (+) x[i,cols-1] for each
 * of `rows` rows ([RW] state-carrying overload: every tile of the row is
 * folded into one monoid state, then pjoin combines across threads / CTAs).
 *   x      device, rows x cols, dtype RR_F32 or RR_I32, element-aligned
 *          (any 4-byte alignment; 16-byte alignment enables vector loads).
 *   op     RR_OP_SUM, RR_OP_MAX or RR_OP_MIN.
 *   out    device, rows elements of the same dtype as x; must not overlap x.
 * fp32 sum is accumulated in fp32 in a fixed order (result within the
 * usual fp32 summation error); int32 sum wraps modulo 2^32; max / min are
 * exact, with max(+0,-0) = +0, min(+0,-0) = -0 and NaN propagating as the
 * quiet NaN 0x7fc00000.  cols == 0 writes the identity (0, -inf / INT_MIN,
 * +inf / INT_MAX).  The tier is picked from rows, cols and the SM count:
 * cols <= 32 tiled, except 16 and 29..32 warp (a thread per row for the
 * other widths up to 32; rows of up to 8 16-byte vectors are read as
 * vectors); cols < 4096 and rows >= SMs warp (a
 * warp segment per row, lanes striding it); rows < SMs and cols >= 4096
 * split-K with C the smallest power of two >= 2 such that rows * C >= SMs,
 * capped at 16 and at the largest cluster the device can co-schedule;
 * otherwise block.
 * Errors: RR_ERR_INVALID (null pointer with rows > 0, negative sizes, bad
 * op / dtype, overlap), RR_ERR_UNSUPPORTED, RR_ERR_CUDA.
 */
int rr_reduce(const void *x, int64_t rows, int64_t cols, int op, int dtype,
              void *out, void *stream);

/* rr_reduce with options (forced tier, cluster size, tile width, per-rank
 * output).  opts may be NULL (same as rr_reduce).  A forced cluster size
 * the device cannot co-schedule returns RR_ERR_UNSUPPORTED. */
int rr_reduce_ex(const void *x, int64_t rows, int64_t cols, int op, int dtype,
                 void *out, void *stream, const rr_reduce_opts *opts);

/*
 * rr_reduce_splitk_multi -- the split-K tier with several clusters per row,
 * for rows too few to cover the GPU with one cluster each ([RW] split-K
 * tier; [CA] within each cluster).  The row is cut into G * C slices; the G
 * clusters of C CTAs of a row each fold C consecutive slices and combine
 * them through distributed shared memory; the cluster results go to
 * `workspace` (rows * G elements of the output type) and a second kernel
 * folds each row's G partials in order.  Deterministic like every tier.
 *   cluster_size      0 = largest the device co-schedules (<= 16), else
 *                     1, 2, 4, 8 or 16.
 *   clusters_per_row  G; 0 = enough that every SM gets a CTA
 *                     (ceil(SMs / (rows * C))), at most 1024.
 *   workspace         device, at least rows * G * 4 bytes (G as resolved;
 *                     rows * 1024 * 4 always suffices), caller-owned, not
 *                     overlapping x or out; its contents are scratch.
 * Same arguments and results as rr_reduce otherwise.
 */
int rr_reduce_splitk_multi(const void *x, int64_t rows, int64_t cols, int op,
                           int dtype, void *out, int cluster_size,
                           int clusters_per_row, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * rr_reduce_axis -- reduction over a non-last axis ([RW] Args: row_coords
 * pins every dimension but ctx.axis, the reduce axis).  x is viewed as a
 * dense row-major [outer][axis][inner] array and
 *   out[o * inner + i] = x[o,0,i] (+) x[o,1,i] (+) ... (+) x[o,axis-1,i].
 *   x      device, outer * axis * inner elements of dtype RR_F32 or RR_I32,
 *          4-byte aligned (16-byte alignment with inner % 4 == 0 enables
 *          128-bit loads).
 *   out    device, outer * inner elements of the same dtype; must not
 *          overlap x.
 * Same element rules as rr_reduce (fp32 sum accumulated in fp32 in a fixed
 * order, int32 sum wraps, max / min exact with the same signed-zero and NaN
 * rules); axis == 0 writes the identity.  inner == 1 is the last-axis
 * reduction and runs rr_reduce's tiers on (rows = outer, cols = axis).
 * For inner > 1 the tiers are laid over the strided rows x[o,:,i]:
 *   RR_TIER_TILED  a thread owns emit_tile_width adjacent rows (1 = the
 *                  serial tier; 2 needs inner even and x 8-byte aligned; 4
 *                  needs inner % 4 == 0 and x 16-byte aligned) and walks the
 *                  axis in order;
 *   RR_TIER_WARP   a warp owns a tile of tile_rows adjacent rows, its lanes
 *                  split the axis and combine with shuffles;
 *   RR_TIER_BLOCK  a CTA owns a tile, its warps split the axis and combine
 *                  in shared memory;
 *   RR_TIER_SPLITK a cluster of cluster_size CTAs owns a tile, each CTA
 *                  folds one chunk of the axis, and each row is folded over
 *                  the CTAs in rank order through distributed shared memory.
 * Block and split-K may also cut each tile's axis into `splits` (G) parts
 * handled by independent CTAs / clusters; their G partial results go to a
 * caller-owned workspace of G * outer * inner * 4 bytes and a second kernel
 * folds them in order g = 0 .. G-1.  rr_reduce_axis itself never splits
 * (it has no workspace); rr_reduce_axis_ex splits when given a workspace,
 * automatically when the shape has too few tiles to cover the GPU.
 * Narrow inner widths that are not a multiple of 4 (2, 3, 5, 6, 7) with a
 * 16-byte aligned x and axis * inner % 4 == 0 take a slab form of the warp
 * tier (16 or more slabs x[o, :, :] per SM: a warp per slab) or of the block
 * tier (2 to 15 per SM: a CTA per slab), reported with tile_rows = inner: the
 * contiguous slab is read with 16-byte loads, element e of each group of 4
 * axis positions folded into column e % inner.
 * The automatic choice is rr_plan_reduce_axis's.
 * Errors: RR_ERR_INVALID (null pointer with work to do, negative sizes, bad
 * op / dtype / options, overlap, a forced tile width, tile size or split
 * count the shape, alignment or workspace does not allow),
 * RR_ERR_UNSUPPORTED (forced cluster size the device cannot co-schedule),
 * RR_ERR_CUDA.
 */
typedef struct {
    int tier;            /* RR_TIER_AUTO or a forced tier */
    int cluster_size;    /* split-K: 0 = automatic, else 1, 2, 4, 8 or 16 */
    int emit_tile_width; /* tiled: 0 = automatic, else 1, 2 or 4 */
    int tile_rows;       /* warp / block / split-K: 0 = automatic, else a
                            power of two from V to 32 * V, where V = 4 when
                            inner % 4 == 0 and x is 16-byte aligned (128-bit
                            loads), else 1 */
    int splits;          /* block / split-K: 0 = automatic (1 without a
                            workspace), else G >= 1 */
    void *workspace;     /* device scratch for G > 1, caller-owned, not
                            overlapping x or out; contents are scratch */
    size_t workspace_bytes;
} rr_axis_opts;

int rr_reduce_axis(const void *x, int64_t outer, int64_t axis, int64_t inner,
                   int op, int dtype, void *out, void *stream);
int rr_reduce_axis_ex(const void *x, int64_t outer, int64_t axis,
                      int64_t inner, int op, int dtype, void *out,
                      void *stream, const rr_axis_opts *opts);

/* A resolved rr_reduce_axis launch (see rr_plan_reduce_axis). */
typedef struct {
    int tier;               /* RR_TIER_TILED / WARP / BLOCK / SPLITK */
    int cluster_size;       /* split-K CTAs per cluster, else 1 */
    int emit_tile_width;    /* tiled: rows per thread, else 0 */
    int tile_rows;          /* warp / block / split-K: rows per tile, else 0 */
    int splits;             /* G, clusters (or CTAs) per tile */
    size_t workspace_bytes; /* G * outer * inner * 4 when G > 1, else 0 */
} rr_axis_plan;

/*
 * rr_plan_reduce_axis -- the host-only tier choice of rr_reduce_axis_ex for
 * a device with `sm_count` SMs whose largest co-schedulable cluster is
 * `max_cluster` CTAs, x aligned to `x_align` bytes (4, 8 or 16), with
 * (with_workspace != 0) or without a workspace.  inner == 1 reports the
 * last-axis plan of rr_plan_reduce.  Touches no GPU.
 */
int rr_plan_reduce_axis(int64_t outer, int64_t axis, int64_t inner,
                        int sm_count, int max_cluster, int x_align,
                        int with_workspace, rr_axis_plan *plan);

/*
 * rr_reduce_axis_workspace_size -- bytes of workspace the automatic plan of
 * rr_reduce_axis_ex wants on the current device for this shape and x
 * alignment (0: it does not split).  Queries device properties only.
 */
int rr_reduce_axis_workspace_size(int64_t outer, int64_t axis, int64_t inner,
                                  int x_align, size_t *bytes_out);

/*
 * rr_softmax -- out[i,:] = exp(x[i,:] - m_i) / s_i with m_i = max_j x[i,j],
 * s_i = sum_j exp(x[i,j] - m_i) ([RW]: pass 1 reduces the (max, sum)
 * monoid, pass 2 is a stateless map over the row).  The row is read from
 * HBM once when it fits on chip.
 *   x      device, rows x cols, in_dtype RR_BF16 or RR_F32.
 *   out    device fp32, rows x cols; must not overlap x.
 *   cols must be >= 1 (RR_ERR_INVALID otherwise).
 */
int rr_softmax(const void *x, int64_t rows, int64_t cols, int in_dtype,
               float *out, void *stream);

/*
 * rr_layernorm_stats -- per row mean = sum x / cols, population variance
 * var = sum (x - mean)^2 / cols taken about the mean in a second pass over
 * the on-chip row, rstd = 1 / sqrt(var + eps) ([RW]: the statistics reduce
 * that precedes the layernorm rewrite).
 *   x      device, rows x cols, in_dtype RR_BF16 or RR_F32; cols >= 1.
 *   mean, rstd  device fp32, rows elements each.
 */
int rr_layernorm_stats(const void *x, int64_t rows, int64_t cols, int in_dtype,
                       float eps, float *mean, float *rstd, void *stream);

/*
 * Options of rr_softmax_ex / rr_layernorm_stats_ex / rr_layernorm_ex ([RW]
 * tier semantics for the two-pass row operations).  Zero-initialise and set
 * what you need.
 *   tier          RR_TIER_AUTO, RR_TIER_WARP (a segment of lanes_per_row
 *                 lanes of a warp per row, the row in its registers),
 *                 RR_TIER_BLOCK (a CTA per row, the row on chip) or
 *                 RR_TIER_SPLITK (a cluster of C CTAs per row).
 *   cluster_size  split-K: 0 = automatic, else 1, 2, 4, 8 or 16.
 *   lanes_per_row warp tier: 0 = automatic, else 1, 2, 4, 8, 16 or 32.
 * Warp tier: lane j of a row's segment holds the row's 16-byte vectors j,
 * j + L, j + 2L, ... (at most 8 per lane, so rows of up to 256 vectors:
 * 2048 bf16 or 1024 fp32 elements); both reductions of a row are shuffles
 * inside the segment.  This vector form needs cols a multiple of 8 (bf16)
 * or 4 (fp32), x 16-byte aligned, the softmax output 32-byte (bf16 input)
 * or 16-byte (fp32) aligned, and for the layernorm gamma / beta 16-byte and
 * the output 16-byte (bf16 input) or 8-byte (fp32) aligned.  Other rows
 * take a chunked form: a row's whole aligned 16-byte chunks spread over the
 * lanes the same way (at most 256 chunks: 2055 bf16 / 1027 fp32 elements),
 * its head and tail elements (before its first, after its last 16-byte
 * boundary) held by the lanes one by one; gamma / beta of the rewrite are
 * copied into shared memory.  Softmax and the rewrite take it when their
 * output sits at x's offset within a 16-byte chunk (always so for 16-byte
 * aligned bases), the rewrite from 32 elements on; otherwise an
 * element-wise form, lane j holding elements j, j + L, ... (4 per lane
 * below 32 lanes, up to 1024 elements).  A forced warp tier returns
 * RR_ERR_UNSUPPORTED when the row does not fit lanes_per_row lanes (or any
 * form).  AUTO picks it for rows that fit when there are at least 4 rows
 * per SM (8 for rr_layernorm), with about 4 vectors or chunks per lane (2
 * for rows of up to 8 and for rr_layernorm; a lane per row for rows of up
 * to 2).  The statistics of rr_layernorm and rr_layernorm_stats on the same
 * x are bitwise equal when both take the same form and lanes.
 * Split-K: CTA r owns slice r of the row, and the row takes two cluster
 * combines ([CA]) on two slots without a tail sync between them: softmax
 * combines the CTA maxima, then the CTA sums rescaled to the row max (one
 * read of the slice for both); layernorm combines the sums, then the
 * squared deviations about the mean.  Every CTA folds in rank order, so
 * every CTA holds the same row statistics.  AUTO picks split-K when
 * rows < SMs and cols >= 16384, with C the smallest power of two >= 2 such
 * that rows * C >= SMs, at most 16.
 * Staged rows: with rows >= SMs, aligned rows beyond the register form
 * (softmax: more than 1024 16-byte vectors, i.e. 8192 bf16 / 4096 fp32
 * elements; layernorm: more than 2048) are copied into shared memory with
 * bulk copies and read from there by every pass, one HBM read per element:
 * a CTA per row while a row fits 96 KiB, else the smallest cluster (<= 16)
 * whose slices do, each CTA staging its slice (reported as the split-K tier
 * of that cluster size); the statistics stage only up to clusters of 4.
 * Rows that are not 16-byte aligned (a width that is not a vector multiple,
 * or a misaligned operand) and too few or too long for the warp tier are
 * staged too, beyond 32 vectors for softmax, 1024 for the statistics, 2048
 * for rr_layernorm, with their partial first and last 16-byte chunks loaded
 * element by element.  Below that, the statistics and rr_layernorm hold
 * such rows (up to 1024 vectors) at a CTA per row in registers as their
 * head elements, whole 16-byte vectors and tail elements (the chunked
 * form; the rewrite reads gamma / beta from a copy each CTA keeps in
 * shared memory, (cols + cols / 8 + 1) * 8 bytes for bf16 input, cols / 4
 * for fp32), where 8-byte aligned rows do not take the register form in
 * 8-byte vectors; rr_layernorm takes the scalar form for its rows of 1025
 * to 2048 vectors.  rr_softmax takes the chunked form for rows of up to
 * 4096 elements whose output shares x's offset within a 16-byte chunk
 * (always so for a 16-byte aligned x and output), and stages the rest.
 * Long rows that are not staged take split-K over global memory with
 * slices of at most 128 KiB.  A forced block tier stages when it applies; a
 * forced split-K tier reads from global memory.
 * Grid form (given a workspace): split-K whose G slices per row go to the
 * CTAs of a plain grid rather than a cluster, so that a few rows cover
 * every SM.  One kernel folds each slice into its partial state (softmax:
 * the (max, sum) pair; layernorm: (count, mean, M2)) and stores it in the
 * workspace; a second kernel, in stream order, folds each row's G states
 * in one fixed order and writes the row's result (softmax and the rewrite
 * read the slice again).  AUTO takes it, when a workspace of
 * rr_rowwise_workspace_size bytes is given, for fewer rows than SMs of at
 * least 16384 elements, x 16-byte aligned, cols a multiple of 8, the
 * softmax output 32-byte and the rewrite's output, gamma and beta 16-byte
 * aligned; G = about 4 CTAs per SM over all rows (slices of at least 2048
 * elements, G <= 1024).  Forced with tier RR_TIER_SPLITK, cluster_size 0
 * or 1 and splits = G.  The statistics of rr_layernorm and
 * rr_layernorm_stats in this form are bitwise equal for the same G.
 * Two-pass form of rr_layernorm (given a workspace): for at least as many
 * rows as SMs, rows of at least 256 KiB of x, aligned as for the grid form,
 * the statistics are streamed through the shared-memory ring (a CTA per
 * row, as rr_layernorm_stats takes them, so their bits are the same) into
 * mean / rstd where asked for, else into the workspace; a second kernel
 * reads x again and writes y, each thread holding gamma / beta for its 8
 * columns over a group of rows.  Two HBM reads of x, against the staged
 * form's one, but gamma / beta are no longer reloaded (8 bytes an element)
 * for every row.
 *   splits          0 = automatic, else G (1..1024) CTAs per row.
 *   workspace       device scratch, 16-byte aligned, caller-owned, not
 *                   overlapping any operand, or NULL (no grid form); its
 *                   contents are scratch.  Calls that may run at the same
 *                   time (other streams) need workspaces of their own.
 *   workspace_bytes its size; at least rows * G * 16 for the grid form (a
 *                   16-byte state per CTA), rows * 8 for the two-pass form
 *                   (a row's mean and rstd); the automatic plan does
 *                   without either form when it is smaller.
 */
typedef struct {
    int tier;
    int cluster_size;
    int lanes_per_row;
    int splits;
    void *workspace;
    size_t workspace_bytes;
} rr_rowwise_opts;

/*
 * rr_rowwise_workspace_size -- bytes of workspace the automatic plan of
 * rr_softmax_ex / rr_layernorm_stats_ex / rr_layernorm_ex wants on the
 * current device for rows x cols of in_dtype with aligned operands (0: it
 * takes neither the grid nor the two-pass form).  Queries device
 * properties only.
 */
int rr_rowwise_workspace_size(int64_t rows, int64_t cols, int in_dtype,
                              int row_op, size_t *bytes_out);

/* rr_softmax with options; opts may be NULL.  RR_ERR_UNSUPPORTED if a
 * forced cluster size cannot be co-scheduled. */
int rr_softmax_ex(const void *x, int64_t rows, int64_t cols, int in_dtype,
                  float *out, void *stream, const rr_rowwise_opts *opts);

/* rr_layernorm_stats with options; opts may be NULL. */
int rr_layernorm_stats_ex(const void *x, int64_t rows, int64_t cols,
                          int in_dtype, float eps, float *mean, float *rstd,
                          void *stream, const rr_rowwise_opts *opts);

/*
 * rr_layernorm -- the layernorm rewrite fused with its statistics ([RW]: the
 * map pass that follows the statistics reduce):
 *   out[i,j] = bf16_rn((x[i,j] - mean_i) * rstd_i * gamma[j] + beta[j])
 * with mean_i, rstd_i as in rr_layernorm_stats.  The row is read from HBM
 * once when it fits on chip.
 *   x        device, rows x cols, in_dtype RR_BF16 or RR_F32; cols >= 1.
 *   gamma, beta  device fp32, cols elements each.
 *   out_bf16 device, rows x cols bf16 bit patterns; must not overlap x.
 *   mean, rstd   device fp32 rows elements each, or NULL if not wanted.
 */
int rr_layernorm(const void *x, int64_t rows, int64_t cols, int in_dtype,
                 float eps, const float *gamma, const float *beta,
                 uint16_t *out_bf16, float *mean, float *rstd, void *stream);

/* rr_layernorm with options (warp, block or split-K tier); opts may be NULL. */
int rr_layernorm_ex(const void *x, int64_t rows, int64_t cols, int in_dtype,
                    float eps, const float *gamma, const float *beta,
                    uint16_t *out_bf16, float *mean, float *rstd, void *stream,
                    const rr_rowwise_opts *opts);

/*
 * rr_cluster_allreduce -- the [CA] primitive, run `iters` times back to back
 * by `clusters` clusters of `cluster_size` CTAs.  For iteration t, cluster
 * c, rank r, the CTA's block-reduced vector is vals[((t*clusters + c)*C
 * + r)*width + j] (loaded by thread 0 only).  Every CTA gathers every peer's
 * vector through distributed shared memory and folds it in rank order
 * 0..C-1, so all CTAs hold the same bits; res receives each rank's result
 * in the same layout.  two_slot = 0 retires the slot with a trailing
 * cluster barrier after every combine (need_tail_sync = True); two_slot = 1
 * drops it and alternates between two slots ([CA] need_tail_sync).
 * skew_cycles > 0 makes each rank spin a pseudo-random multiple (0..7) of
 * skew_cycles clock cycles before each combine, so that CTAs race ahead.
 * When `mismatches` (device int64) is given, every thread of every CTA also
 * re-folds the inputs of its iteration from global memory in rank order,
 * compares bits with its own result and adds the number of differing values
 * to *mismatches; with NULL the kernel only runs the combines (for timing).
 *   cluster_size 1..16 (16 needs the device's non-portable cluster size),
 *   width 1, 2, 4 or 8, dtype RR_F32 or RR_I32; iters >= 0 (0 is a no-op);
 *   skew_cycles 0..2^20.
 */
int rr_cluster_allreduce(const void *vals, int clusters, int cluster_size,
                         int width, int op, int dtype, int iters, int two_slot,
                         int64_t skew_cycles, void *res,
                         int64_t *mismatches, void *stream);

/*
 * rr_cluster_allreduce_selftest -- BLOCKING self-test of the [CA]
 * primitive: draws seeded per-rank vectors on the device (a counter-based
 * hash of seed, iteration, cluster, rank, element), runs
 * rr_cluster_allreduce with 2 clusters of `cluster_size` CTAs and a rank
 * skew, synchronises, and writes to *mismatches_out (host pointer) the
 * number of values, over all threads and iterations, that differ in bits
 * from the rank-order fold.  Returns RR_OK, or RR_ERR_MISMATCH when the
 * count is non-zero.  Allocates and frees its own device scratch.
 */
int rr_cluster_allreduce_selftest(int cluster_size, int width, int op,
                                  int dtype, int iters, int two_slot,
                                  uint64_t seed, void *stream,
                                  int64_t *mismatches_out);

/*
 * rr_cluster_allreduce_selftest_ex -- rr_cluster_allreduce_selftest that
 * also hands the run back for a check on the host ([CA] description: every
 * CTA folds every rank's vector in rank order, so the host can redo that
 * fold from the inputs and compare bits with every rank's result).
 *   vals_host  host buffer of n = iters * 2 * cluster_size * width 32-bit
 *              values, or NULL: receives the seeded per-rank inputs, laid
 *              out [iters][2 clusters][cluster_size][width].  Value i is
 *              u = splitmix64(seed ^ splitmix64(i)) (splitmix64 as published
 *              by Steele, Lea and Flood, "Fast splittable pseudorandom number
 *              generators", 2014); int32: the high 32 bits of u; fp32:
 *              ldexp((u >> 40) * 2^-23 - 1, (u >> 8) % 41 - 20).
 *   res_host   host buffer of n values, or NULL: receives every rank's
 *              combined result (thread 0's copy) in the same layout.
 * Both are written only when the call returns RR_OK or RR_ERR_MISMATCH.
 * Otherwise as rr_cluster_allreduce_selftest.
 */
int rr_cluster_allreduce_selftest_ex(int cluster_size, int width, int op,
                                     int dtype, int iters, int two_slot,
                                     uint64_t seed, void *stream,
                                     int64_t *mismatches_out, void *vals_host,
                                     void *res_host);

/*
 * rr_cluster_allreduce_selftest_noalloc -- the same blocking self-test as
 * rr_cluster_allreduce_selftest (same arguments, same checks, same result),
 * but it allocates no device memory: no cudaMalloc, no cudaFree, no
 * allocating library call.  The pages have no counterpart of this entry
 * point; it exists for callers that cannot allocate, such as a serving
 * process whose memory pool already holds the whole device, or one that
 * must not risk the implicit device synchronisation of cudaMalloc/cudaFree
 * between its own kernels.
 *   Scratch: a fixed device array inside librr.so, 2 * 2^18 32-bit values
 *   plus a counter (about 2 MiB).  Every GPU that loads the library holds it
 *   until the process exits.  iters * 2 * cluster_size * width must not
 *   exceed 2^18 (262144); larger requests return RR_ERR_INVALID.
 *   The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.  Each call resets the counter it needs; the array keeps
 *   the last call's other contents.  All calls share the one array: calls
 *   from several host threads of a process run one after another (each holds
 *   a process-wide lock for its whole, blocking, duration, and waits for
 *   its stream before it returns, on failure too).
 * Returns RR_OK, RR_ERR_MISMATCH, RR_ERR_INVALID, RR_ERR_UNSUPPORTED or
 * RR_ERR_CUDA.
 */
int rr_cluster_allreduce_selftest_noalloc(int cluster_size, int width, int op,
                                          int dtype, int iters, int two_slot,
                                          uint64_t seed, void *stream,
                                          int64_t *mismatches_out);

/*
 * rr_cluster_allreduce_selftest_noalloc_ex -- the no-allocation self-test
 * that also copies its inputs and every rank's results out of the fixed
 * array into caller-owned host buffers (vals_host, res_host: n 32-bit values
 * each, or NULL; layout and values as rr_cluster_allreduce_selftest_ex), so
 * that a caller can check the run on the host.  Allocates nothing, like
 * rr_cluster_allreduce_selftest_noalloc; the pages have no counterpart.
 */
int rr_cluster_allreduce_selftest_noalloc_ex(int cluster_size, int width,
                                             int op, int dtype, int iters,
                                             int two_slot, uint64_t seed,
                                             void *stream,
                                             int64_t *mismatches_out,
                                             void *vals_host, void *res_host);

/*
 * rr_splitk_combine -- split-K attention-output combine ([FA]).
 *   O       device fp32 [P][rows][D] partial outputs (unnormalised).
 *   m, l    device fp32 [P][rows] per-partition row max (raw scores) and
 *           row sum of exp.
 *   out_bf16 device [rows][D] bf16 bit patterns.
 * Per row: M = max_p m_p, w_p = exp2((m_p - M) * scale_log2e),
 * L = sum_p w_p l_p (rank order), out = bf16_rn(sum_p w_p O_p / L); rows
 * with M = -inf or L = 0 are written as +0.  In the page's design a cluster
 * of P CTAs handles a tile of rows: CTA p stages its own partial into its
 * shared memory, publishes it with a cluster barrier, then folds the P
 * partials of its column band [p*D/P, (p+1)*D/P) in rank order through
 * distributed shared memory and stores that band; a partition whose band is
 * empty (D < P) only stages and publishes.  This call takes the fastest
 * variant the arguments allow (RR_COMBINE_AUTO of rr_splitk_combine_ex);
 * every variant returns the same bits.
 *   P in 1..16 (16 needs the non-portable cluster size), D in 1..1024.
 * Errors: RR_ERR_INVALID, RR_ERR_UNSUPPORTED (cluster of P CTAs cannot be
 * co-scheduled), RR_ERR_CUDA.  A staging copy that does not land within the
 * device wait budget sets the device error word (see rr_device_status).
 */
int rr_splitk_combine(const float *O, const float *m, const float *l, int P,
                      int64_t rows, int D, float scale_log2e,
                      uint16_t *out_bf16, void *stream);

/* Combine variants (all compute the same result; see rr_splitk_combine_ex). */
typedef enum {
    RR_COMBINE_AUTO = 0,    /* the fastest variant the arguments allow:
                               direct, else push, else pull, else generic */
    RR_COMBINE_PULL = 1,    /* each CTA reads its depth band of every peer's
                               staged tile through DSMEM ([FA] as printed);
                               P in {1,2,4,8,16}, D % 4P == 0 */
    RR_COMBINE_PUSH = 2,    /* each CTA bulk-copies every peer's row slice of
                               its staged tile into that peer's shared memory
                               (the scatter rides the copy engine); P in
                               {1,2,4,8,16}, D % 4 == 0, D <= 256 */
    RR_COMBINE_GENERIC = 3, /* one tile per cluster, plain loads, any P <= 16
                               and D <= 1024, unequal or empty bands */
    RR_COMBINE_DIRECT = 4   /* no cluster: each CTA stages the rows of all P
                               partitions itself and folds them locally;
                               same DRAM traffic, no exchange between CTAs;
                               P in {1,2,4,8,16}, D % 4 == 0, 2*P*D*4 <= 96 KiB */
} rr_combine_mode;

/*
 * rr_splitk_combine_ex -- rr_splitk_combine with an explicit variant.
 * Every variant stages, publishes across the cluster of P CTAs, folds the P
 * partials in rank order 0..P-1 and stores bf16; they differ in how the
 * partials move between CTAs.  A variant whose conditions the arguments do
 * not meet returns RR_ERR_UNSUPPORTED (AUTO never does for valid
 * arguments).  16-byte aligned O and 8-byte aligned out are required by
 * PULL and PUSH.
 */
int rr_splitk_combine_ex(const float *O, const float *m, const float *l, int P,
                         int64_t rows, int D, float scale_log2e,
                         uint16_t *out_bf16, void *stream, int mode);

/* Synchronises `stream`, then reads and clears the current device's error
 * word: RR_OK, or RR_ERR_TIMEOUT if a bounded device wait gave up since the
 * last call.  RR_ERR_CUDA if the synchronisation itself failed. */
int rr_device_status(void *stream);

/* Tier and width of the last reduce / softmax / layernorm call made by this
 * process: (twopass << 28) | (chunked << 27) | ((width >> 8) << 19) | (grid << 18) |
 * (ring << 17) | (staged << 16) | ((width & 0xff) << 8) | tier, width the
 * cluster size
 * (the warp tier of the row operations: lanes per row; the grid form: CTAs
 * per row), staged 1 when a row operation staged its rows in shared
 * memory, ring 1 when it streamed them through a shared-memory ring of bulk
 * copies (one combine per row; the layernorm statistics as a (count, mean,
 * M2) monoid), grid 1 when it took the grid form (rr_rowwise_opts), chunked
 * 1 when a row operation held a row that is not 16-byte aligned in
 * registers as its head, whole 16-byte vectors and tail (a CTA per row),
 * twopass 1 when rr_layernorm took its two-pass form. */
int rr_last_tier(void);

/* Static English name of a status code. */
const char *rr_status_string(int status);

/*
 * rr_plan_reduce -- the host-only tier choice of rr_reduce for a device
 * with `sm_count` SMs whose largest co-schedulable cluster is
 * `max_cluster` CTAs: writes the tier and cluster size rr_reduce would use.
 * Touches no GPU.  Returns RR_ERR_INVALID on negative sizes.
 */
int rr_plan_reduce(int64_t rows, int64_t cols, int sm_count, int max_cluster,
                   int *tier_out, int *cluster_out);

/* The two-pass row operations, for rr_plan_rowwise. */
typedef enum { RR_ROW_SOFTMAX = 0, RR_ROW_LNSTATS = 1, RR_ROW_LAYERNORM = 2 } rr_row_op;

/*
 * rr_plan_rowwise -- the host-only tier choice of rr_softmax (row_op
 * RR_ROW_SOFTMAX), rr_layernorm_stats (RR_ROW_LNSTATS) or rr_layernorm
 * (RR_ROW_LAYERNORM) with automatic options ([RW] tier semantics), for a
 * device with `sm_count` SMs whose largest co-schedulable cluster is
 * `max_cluster` CTAs.  `aligned` != 0 says every operand meets the warp
 * tier's alignment (rr_rowwise_opts); cols must also be a multiple of the
 * 16-byte vector.  Rows that are not are planned for operands whose bases
 * are 16-byte aligned (the outputs then share x's offset within a chunk).
 * Writes the tier and its width: lanes per row (warp),
 * cluster size (split-K) or 1 (block); *staged_out (if not NULL) 1 when the
 * block / split-K tier stages the rows in shared memory, 2 when it streams
 * them through a shared-memory ring (the split-K width is then the cluster
 * size planned; a launch may take a smaller one, down to 2, when the device
 * cannot co-schedule a cluster that size for every row), 3 for the grid
 * form (split-K, width = G CTAs per row), which the plan considers only
 * with with_workspace != 0, 4 for the chunked register form of rows that
 * are not 16-byte aligned (the statistics and the rewrite up to 1024
 * vectors, softmax up to 4096 elements), 5 for rr_layernorm's two-pass
 * form (with_workspace != 0 only).  Touches no GPU.  RR_ERR_INVALID on negative
 * sizes, sm_count or max_cluster < 1, a bad dtype or row_op.
 */
int rr_plan_rowwise(int64_t rows, int64_t cols, int in_dtype, int row_op,
                    int aligned, int sm_count, int max_cluster,
                    int with_workspace, int *tier_out, int *width_out,
                    int *staged_out);

/*
 * rr_test_wait_timeout -- failure-detection hook: launches one CTA that
 * waits on a shared-memory mbarrier that nothing completes, with a budget
 * of `budget_iters` polls.  The wait gives up, sets the device error word
 * and the kernel returns normally, so a following rr_device_status
 * reports RR_ERR_TIMEOUT and the context stays usable.
 */
int rr_test_wait_timeout(int64_t budget_iters, void *stream);

/*
 * rr_test_inject_error -- failure-injection hook: the next `count` calls
 * that would enqueue work validate their arguments and then return
 * RR_ERR_CUDA, as if the CUDA runtime had refused them, without touching
 * the device; later calls run normally.  count 0 clears a pending count.
 * Returns RR_ERR_INVALID for count < 0.
 */
int rr_test_inject_error(int count);

#ifdef __cplusplus
}
#endif

#endif /* RR_H_ */
