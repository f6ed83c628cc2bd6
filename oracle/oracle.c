/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the row-reduction
 * hot path.  TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under cluster_reductions_gb300/) never calls into it, and the
 * two share no code, headers, tables or constants.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math), so every
 * floating-point operation below is the IEEE operation written in the source.
 *
 * Every function is serial per row and computes the plain definition of the
 * result in fp64 (fp32 / int32 where the definition itself is an fp32 or
 * int32 fold).  Sources:
 *   - "cluster_allreduce" (Mojo API page, max/gpu/primitives/cluster):
 *     description and the combine_fn / cluster_size parameters -- the
 *     cross-CTA fold is taken in rank order; with one CTA it is a broadcast.
 *   - "reduce" (Mojo API page, algorithm/gpu/rowwise): the row-wise monoid
 *     reduction over the reduce axis; softmax pass 2 and the layernorm
 *     rewrite named there as the two-pass users.
 *   - "fa4_splitk_reduce_scatter_write" (Mojo API page, sm100 softmax_warp):
 *     the split-K output combine -- per-partition (max, sum) statistics,
 *     exp2 rescaling by scale_log2e, weighted sum of partial outputs, bf16
 *     store.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - max/min of +0 and -0: max gives +0, min gives -0, whatever the order;
 *     any NaN operand gives NaN (the quiet NaN 0x7fc00000 for fp32).
 *   - int32 sum wraps modulo 2^32 (two's complement).
 *   - layernorm variance is the population variance (divide by N), computed
 *     about the mean in a second pass; eps is added inside the square root.
 *   - combine: m_p are raw scores; the scale multiplies the difference
 *     (m_p - M); a row whose M is -inf or whose L is 0 is written as +0.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Operation codes of this oracle (its own numbering, defined here). */
enum { ORC_SUM = 0, ORC_MAX = 1, ORC_MIN = 2 };

/* ------------------------------------------------------------------ */
/* scalar helpers                                                      */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* fp32 max with the +0/-0 and NaN reading stated in the header. */
static float orc_fmax(float a, float b)
{
    if (a != a || b != b) return bits_f32(0x7fc00000u);
    if (a > b) return a;
    if (b > a) return b;
    /* equal: only +0 / -0 can differ in bits; +0 wins */
    return bits_f32(f32_bits(a) & f32_bits(b));
}

static float orc_fmin(float a, float b)
{
    if (a != a || b != b) return bits_f32(0x7fc00000u);
    if (a < b) return a;
    if (b < a) return b;
    /* equal: -0 wins */
    return bits_f32(f32_bits(a) | f32_bits(b));
}

/* bf16 (stored as its 16 high bits of an fp32) widened exactly to double. */
static double bf16_to_f64(uint16_t h)
{
    return (double)bits_f32(((uint32_t)h) << 16);
}

/*
 * double -> bf16, round to nearest, ties to even, directly from the double
 * (no intermediate fp32 rounding, which could round twice).
 * bf16 keeps 8 significant bits and fp32's exponent range; its subnormals
 * are spaced 2^-133 apart.
 */
uint16_t oracle_f64_to_bf16(double x)
{
    if (x != x) return 0x7fc0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    if (isinf(ax)) return (uint16_t)(sign | 0x7f80u);
    int e;                       /* ax = f * 2^e, f in [0.5, 1) */
    frexp(ax, &e);
    int k = e - 1;               /* ax in [2^k, 2^(k+1)) */
    if (k < -126) k = -126;      /* subnormal range: fixed spacing */
    double ulp = ldexp(1.0, k - 7);
    double q = rint(ax / ulp);   /* default rounding mode: nearest-even */
    double r = q * ulp;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7f80u);
    float rf = (float)r;         /* exact: r has <= 8 significant bits */
    return (uint16_t)(sign | (f32_bits(rf) >> 16));
}

/* ------------------------------------------------------------------ */
/* row reductions ("reduce" page: the state-carrying overload folds   */
/* every element of the row into one monoid state)                    */
/* ------------------------------------------------------------------ */

/*
 * fp32 rows.  op = sum: out[r] = sum_i (double)x[r,i], accumulated in fp64
 * in index order.  op = max / min: the exact fp32 result, widened to double
 * (so its sign and NaN-ness survive).  cols == 0 gives the identity
 * (0, -inf, +inf).
 */
void oracle_reduce_f32(const float *x, int64_t rows, int64_t cols, int op,
                       double *out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *row = x + r * cols;
        if (op == ORC_SUM) {
            double acc = 0.0;
            for (int64_t i = 0; i < cols; ++i) acc += (double)row[i];
            out[r] = acc;
        } else if (op == ORC_MAX) {
            float acc = -INFINITY;
            for (int64_t i = 0; i < cols; ++i) acc = orc_fmax(acc, row[i]);
            out[r] = (double)acc;
        } else {
            float acc = INFINITY;
            for (int64_t i = 0; i < cols; ++i) acc = orc_fmin(acc, row[i]);
            out[r] = (double)acc;
        }
    }
}

/* int32 rows: sum wraps modulo 2^32; max / min are exact.  Identity for
 * cols == 0: 0, INT32_MIN, INT32_MAX. */
void oracle_reduce_i32(const int32_t *x, int64_t rows, int64_t cols, int op,
                       int32_t *out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t *row = x + r * cols;
        if (op == ORC_SUM) {
            uint32_t acc = 0u;
            for (int64_t i = 0; i < cols; ++i) acc += (uint32_t)row[i];
            out[r] = (int32_t)acc;
        } else if (op == ORC_MAX) {
            int32_t acc = INT32_MIN;
            for (int64_t i = 0; i < cols; ++i) if (row[i] > acc) acc = row[i];
            out[r] = acc;
        } else {
            int32_t acc = INT32_MAX;
            for (int64_t i = 0; i < cols; ++i) if (row[i] < acc) acc = row[i];
            out[r] = acc;
        }
    }
}

/*
 * Reduction over a non-last axis ("reduce" page: row_coords pins every
 * dimension but ctx.axis, the reduce axis).  x is [outer][axis][inner],
 * dense; out[o][i] folds x[o][0][i], x[o][1][i], ... in axis order, with the
 * same element types and rules as oracle_reduce_f32 / oracle_reduce_i32
 * (out is double for fp32 input, int32 for int32 input).  dtype: 0 = fp32,
 * 1 = int32.
 */
void oracle_reduce_axis(const void *x, int64_t outer, int64_t axis, int64_t inner,
                        int op, int dtype, void *out)
{
    for (int64_t o = 0; o < outer; ++o) {
        for (int64_t i = 0; i < inner; ++i) {
            if (dtype == 0) {
                const float *xf = (const float *)x;
                double s = 0.0;
                float m = (op == ORC_MAX) ? -INFINITY : INFINITY;
                for (int64_t a = 0; a < axis; ++a) {
                    float v = xf[(o * axis + a) * inner + i];
                    if (op == ORC_SUM) s += (double)v;
                    else if (op == ORC_MAX) m = orc_fmax(m, v);
                    else m = orc_fmin(m, v);
                }
                ((double *)out)[o * inner + i] = (op == ORC_SUM) ? s : (double)m;
            } else {
                const int32_t *xi = (const int32_t *)x;
                uint32_t s = 0u;
                int32_t m = (op == ORC_MAX) ? INT32_MIN : INT32_MAX;
                for (int64_t a = 0; a < axis; ++a) {
                    int32_t v = xi[(o * axis + a) * inner + i];
                    if (op == ORC_SUM) s += (uint32_t)v;
                    else if (op == ORC_MAX) { if (v > m) m = v; }
                    else { if (v < m) m = v; }
                }
                ((int32_t *)out)[o * inner + i] = (op == ORC_SUM) ? (int32_t)s : m;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* cluster fold ("cluster_allreduce" page: every CTA folds the peers'  */
/* block-reduced vectors in rank order; cluster_size 1 is a broadcast) */
/* ------------------------------------------------------------------ */

/*
 * vals is [C][W] (rank-major).  out[j] = v_0[j] (+) v_1[j] (+) ... (+)
 * v_{C-1}[j], folded left to right in the element type itself (fp32 or
 * int32), so the result is the exact bit pattern a rank-order fold gives.
 * dtype: 0 = fp32, 1 = int32.
 */
void oracle_cluster_fold(const void *vals, int C, int W, int op, int dtype,
                         void *out)
{
    for (int j = 0; j < W; ++j) {
        if (dtype == 0) {
            const float *v = (const float *)vals;
            float acc = v[j];
            for (int r = 1; r < C; ++r) {
                float b = v[(int64_t)r * W + j];
                if (op == ORC_SUM) acc = acc + b;
                else if (op == ORC_MAX) acc = orc_fmax(acc, b);
                else acc = orc_fmin(acc, b);
            }
            ((float *)out)[j] = acc;
        } else {
            const int32_t *v = (const int32_t *)vals;
            int32_t acc = v[j];
            for (int r = 1; r < C; ++r) {
                int32_t b = v[(int64_t)r * W + j];
                if (op == ORC_SUM) acc = (int32_t)((uint32_t)acc + (uint32_t)b);
                else if (op == ORC_MAX) acc = b > acc ? b : acc;
                else acc = b < acc ? b : acc;
            }
            ((int32_t *)out)[j] = acc;
        }
    }
}

/* ------------------------------------------------------------------ */
/* two-pass softmax ("reduce" page: pass 1 reduces the (max, sum)      */
/* state, pass 2 is a map over the row)                                */
/* ------------------------------------------------------------------ */

/* x_dtype: 0 = fp32, 2 = bf16 (raw 16-bit patterns).  y[r,i] in fp64:
 * m = max_i x, s = sum_i exp(x_i - m), y_i = exp(x_i - m) / s. */
void oracle_softmax(const void *x, int x_dtype, int64_t rows, int64_t cols,
                    double *y)
{
    for (int64_t r = 0; r < rows; ++r) {
        double *yr = y + r * cols;
        for (int64_t i = 0; i < cols; ++i) {
            yr[i] = (x_dtype == 2)
                ? bf16_to_f64(((const uint16_t *)x)[r * cols + i])
                : (double)((const float *)x)[r * cols + i];
        }
        double m = -INFINITY;
        for (int64_t i = 0; i < cols; ++i) if (yr[i] > m) m = yr[i];
        double s = 0.0;
        for (int64_t i = 0; i < cols; ++i) s += exp(yr[i] - m);
        for (int64_t i = 0; i < cols; ++i) yr[i] = exp(yr[i] - m) / s;
    }
}

/* ------------------------------------------------------------------ */
/* layernorm statistics ("reduce" page: the layernorm rewrite is a     */
/* second pass after the statistics reduce)                            */
/* ------------------------------------------------------------------ */

/* mean = sum x / N; var = sum (x - mean)^2 / N; rstd = 1 / sqrt(var + eps),
 * all in fp64 over the exactly widened inputs. */
void oracle_layernorm_stats(const void *x, int x_dtype, int64_t rows,
                            int64_t cols, double eps, double *mean,
                            double *var, double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t i = 0; i < cols; ++i) {
            s += (x_dtype == 2)
                ? bf16_to_f64(((const uint16_t *)x)[r * cols + i])
                : (double)((const float *)x)[r * cols + i];
        }
        double mu = s / (double)cols;
        double q = 0.0;
        for (int64_t i = 0; i < cols; ++i) {
            double v = (x_dtype == 2)
                ? bf16_to_f64(((const uint16_t *)x)[r * cols + i])
                : (double)((const float *)x)[r * cols + i];
            q += (v - mu) * (v - mu);
        }
        double va = q / (double)cols;
        mean[r] = mu;
        var[r] = va;
        rstd[r] = 1.0 / sqrt(va + eps);
    }
}

/*
 * Layernorm rewrite ("reduce" page: the second, map-style pass after the
 * statistics reduce): y[r,i] = (x[r,i] - mean_r) * rstd_r * gamma[i] + beta[i]
 * in fp64 with the fp64 statistics above, then rounded once to bf16
 * (nearest-even).  y_f64 (optional) receives the unrounded values; mean and
 * rstd (optional) the statistics.
 */
void oracle_layernorm(const void *x, int x_dtype, int64_t rows, int64_t cols,
                      double eps, const float *gamma, const float *beta,
                      double *y_f64, uint16_t *y_bf16, double *mean,
                      double *rstd)
{
    for (int64_t r = 0; r < rows; ++r) {
        double mu, va, rs;
        const char *row = (const char *)x + r * cols * (x_dtype == 2 ? 2 : 4);
        oracle_layernorm_stats(row, x_dtype, 1, cols, eps, &mu, &va, &rs);
        for (int64_t i = 0; i < cols; ++i) {
            double v = (x_dtype == 2)
                ? bf16_to_f64(((const uint16_t *)row)[i])
                : (double)((const float *)row)[i];
            double yv = (v - mu) * rs * (double)gamma[i] + (double)beta[i];
            if (y_f64) y_f64[r * cols + i] = yv;
            if (y_bf16) y_bf16[r * cols + i] = oracle_f64_to_bf16(yv);
        }
        if (mean) mean[r] = mu;
        if (rstd) rstd[r] = rs;
    }
}

/* ------------------------------------------------------------------ */
/* split-K attention-output combine ("fa4_splitk_reduce_scatter_write" */
/* page: partials O_p with statistics (m_p, l_p) are rescaled by       */
/* exp2((m_p - M) * scale_log2e), summed, normalised and stored bf16)  */
/* ------------------------------------------------------------------ */

/*
 * O is [P][rows][D], m and l are [P][rows].  For each row:
 *   M   = max_p m_p
 *   w_p = 2^((m_p - M) * s),  s = (double)scale_log2e
 *   L   = sum_p w_p l_p
 *   out = sum_p w_p O_p / L
 * in fp64, then rounded once to bf16 (nearest-even).  out_f64 (optional,
 * may be NULL) receives the unrounded fp64 value.  A row with M = -inf or
 * L = 0 is written as +0.
 */
void oracle_splitk_combine(const float *O, const float *m, const float *l,
                           int P, int64_t rows, int D, float scale_log2e,
                           double *out_f64, uint16_t *out_bf16)
{
    double s = (double)scale_log2e;
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < P; ++p) {
            double mp = (double)m[(int64_t)p * rows + r];
            if (mp > M) M = mp;
        }
        double L = 0.0;
        double w[64];
        for (int p = 0; p < P; ++p) {
            double mp = (double)m[(int64_t)p * rows + r];
            w[p] = (M == -INFINITY) ? 0.0 : exp2((mp - M) * s);
            L += w[p] * (double)l[(int64_t)p * rows + r];
        }
        int dead = (M == -INFINITY) || (L == 0.0);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int p = 0; p < P; ++p)
                acc += w[p] * (double)O[((int64_t)p * rows + r) * D + d];
            double v = dead ? 0.0 : acc / L;
            if (out_f64) out_f64[r * D + d] = v;
            if (out_bf16) out_bf16[r * D + d] = oracle_f64_to_bf16(v);
        }
    }
}
