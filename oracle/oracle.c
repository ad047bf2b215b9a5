/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the wide-row reduce-then-reuse
 * operators (row softmax, LayerNorm, RMSNorm, int8 quantization, weighted
 * standardization, Pearson correlation).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it is used by the tests, by the package smoke check and by
 * the CPU-baseline leg of the benchmark.  It shares no code, header, constant
 * or helper with the CUDA library.
 *
 * Source of the operators.  The CREDIT summary page ("CREDIT: Cost-guided
 * Reduction-reuse with Efficient DSMEM Inter-CTA Tiling", arXiv 2609.01864v1),
 * section "B. Reduction-Reuse Transformation", models a row as per-element
 * inputs that feed scalar reductions, after which an elementwise function h
 * produces every output element.  The clustered transformation (section
 * "C. Cluster Reduction and Reuse Protocol") only changes where the partial
 * statistics live; the outputs are those of the plain definitions below
 * ("D. Traffic Validation": output traffic and h are unchanged).  So the
 * oracle is the textbook definition of each operator, written out row by
 * row, two passes per statistic, every sum in fp64 in column order:
 *
 *   softmax   m = max_j x_j,  s = sum_j exp(x_j - m),  y_j = exp(x_j - m) / s
 *   LayerNorm mu = sum_j x_j / N,  var = sum_j (x_j - mu)^2 / N   (biased)
 *             y_j = (x_j - mu) / sqrt(var + eps) * gamma_j + beta_j
 *   RMSNorm   ms = sum_j x_j^2 / N,  y_j = x_j / sqrt(ms + eps) * w_j
 *
 * gamma / beta / w absent (NULL) mean gamma = 1, beta = 0, w = 1.
 *
 * Readings where the pages are silent: the variance is biased (divide by N)
 * and eps sits inside the square root for both norms; RMSNorm is not on the
 * pages and follows the usual definition above.
 *
 * Inputs are the exact bytes the GPU receives: dtype 0 = fp32, 1 = bf16
 * (raw 16-bit patterns), 2 = fp64.  Every widening to double is exact.
 * Outputs are fp64; no rounding to the GPU's output type happens here.
 *
 * Build: gcc -O2 -fPIC -shared (no -ffast-math: the order and rounding of
 * every operation is the one written).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2

#define OR_OK 0
#define OR_BAD_ARG 1

/* Widen element i of a typed buffer to double.  bf16 is the upper half of an
 * IEEE-754 binary32 word, so its value is that word with 16 zero low bits. */
static double or_load(const void *p, int dtype, int64_t i)
{
    if (dtype == OR_F32) {
        float f;
        memcpy(&f, (const unsigned char *)p + 4 * i, 4);
        return (double)f;
    }
    if (dtype == OR_BF16) {
        uint16_t h;
        uint32_t u;
        float f;
        memcpy(&h, (const unsigned char *)p + 2 * i, 2);
        u = ((uint32_t)h) << 16;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    {
        double d;
        memcpy(&d, (const unsigned char *)p + 8 * i, 8);
        return d;
    }
}

static int or_dtype_ok(int dtype)
{
    return dtype == OR_F32 || dtype == OR_BF16 || dtype == OR_F64;
}

/* Decode n elements of a typed buffer into doubles (used by the tests to read
 * back bf16 / fp32 bytes through the same widening the oracle uses). */
int oracle_widen(const void *x, int dtype, int64_t n, double *out)
{
    int64_t i;
    if (!x || !out || n < 0 || !or_dtype_ok(dtype))
        return OR_BAD_ARG;
    for (i = 0; i < n; ++i)
        out[i] = or_load(x, dtype, i);
    return OR_OK;
}

/* Row softmax over `rows` rows of `cols` contiguous elements. */
int oracle_softmax(const void *x, int dtype, int64_t rows, int64_t cols,
                   double *y)
{
    int64_t r, j;
    if (!x || !y || rows < 0 || cols <= 0 || !or_dtype_ok(dtype))
        return OR_BAD_ARG;
    for (r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        double m = -INFINITY, s = 0.0;
        for (j = 0; j < cols; ++j) {
            double v = or_load(x, dtype, base + j);
            if (v > m)
                m = v;
        }
        for (j = 0; j < cols; ++j)
            s += exp(or_load(x, dtype, base + j) - m);
        for (j = 0; j < cols; ++j)
            y[base + j] = exp(or_load(x, dtype, base + j) - m) / s;
    }
    return OR_OK;
}

/* Row LayerNorm.  gamma / beta: length-cols vectors of dtype pdtype, or NULL.
 * If z is not NULL it receives the normalised value (x - mu)/sqrt(var + eps)
 * before the affine step (the tests use it to size the cancellation bound). */
int oracle_layernorm(const void *x, int dtype, int64_t rows, int64_t cols,
                     const void *gamma, const void *beta, int pdtype,
                     double eps, double *y, double *z)
{
    int64_t r, j;
    if (!x || !y || rows < 0 || cols <= 0 || !or_dtype_ok(dtype) ||
        ((gamma || beta) && !or_dtype_ok(pdtype)) || !(eps >= 0.0))
        return OR_BAD_ARG;
    for (r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        double sum = 0.0, ssd = 0.0, mu, var, inv;
        for (j = 0; j < cols; ++j)
            sum += or_load(x, dtype, base + j);
        mu = sum / (double)cols;
        for (j = 0; j < cols; ++j) {
            double d = or_load(x, dtype, base + j) - mu;
            ssd += d * d;
        }
        var = ssd / (double)cols;
        inv = 1.0 / sqrt(var + eps);
        for (j = 0; j < cols; ++j) {
            double zj = (or_load(x, dtype, base + j) - mu) * inv;
            double g = gamma ? or_load(gamma, pdtype, j) : 1.0;
            double b = beta ? or_load(beta, pdtype, j) : 0.0;
            if (z)
                z[base + j] = zj;
            y[base + j] = zj * g + b;
        }
    }
    return OR_OK;
}

/* Row RMSNorm.  w: length-cols vector of dtype pdtype, or NULL. */
int oracle_rmsnorm(const void *x, int dtype, int64_t rows, int64_t cols,
                   const void *w, int pdtype, double eps, double *y)
{
    int64_t r, j;
    if (!x || !y || rows < 0 || cols <= 0 || !or_dtype_ok(dtype) ||
        (w && !or_dtype_ok(pdtype)) || !(eps >= 0.0))
        return OR_BAD_ARG;
    for (r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        double ss = 0.0, inv;
        for (j = 0; j < cols; ++j) {
            double v = or_load(x, dtype, base + j);
            ss += v * v;
        }
        inv = 1.0 / sqrt(ss / (double)cols + eps);
        for (j = 0; j < cols; ++j) {
            double g = w ? or_load(w, pdtype, j) : 1.0;
            y[base + j] = or_load(x, dtype, base + j) * inv * g;
        }
    }
    return OR_OK;
}

/*
 * Row-wise symmetric int8 quantization (CREDIT summary page, "B. Workload-by-
 * Workload Scaling" and "D. Traffic Validation": the quantization workload,
 * 9 -> 5 B/element for FP32 input, i.e. a 4-byte read and a 1-byte write).
 * The pages do not spell the codes out; the reading is the textbook one:
 *   amax = max_j |x_j|,  scale = amax / 127,
 *   q_j  = clamp(round_half_even(x_j / scale), -127, 127),
 * with q = 0 and scale = 0 for an all-zero row.  scale and x_j / scale are
 * computed in IEEE single precision (the precision of the GPU kernel), so
 * the integer decision is taken in the same precision on both sides; amax is
 * exact in any precision.
 */
int oracle_quantize(const void *x, int dtype, int64_t rows, int64_t cols,
                    int8_t *q, float *scales)
{
    int64_t r, j;
    if (!x || !q || !scales || rows < 0 || cols <= 0 || !or_dtype_ok(dtype))
        return OR_BAD_ARG;
    for (r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        double amax = 0.0;
        float s;
        for (j = 0; j < cols; ++j) {
            double v = fabs(or_load(x, dtype, base + j));
            if (v > amax)
                amax = v;
        }
        s = (float)amax / 127.0f;
        scales[r] = s;
        for (j = 0; j < cols; ++j) {
            float v = (float)or_load(x, dtype, base + j);
            float c;
            if (s == 0.0f) {
                q[base + j] = 0;
                continue;
            }
            c = rintf(v / s);
            if (c > 127.0f)
                c = 127.0f;
            if (c < -127.0f)
                c = -127.0f;
            q[base + j] = (int8_t)c;
        }
    }
    return OR_OK;
}

/*
 * Row-wise weighted standardization ("weighted variance" workload of the
 * CREDIT summary page, section "B. Workload-by-Workload Scaling").  The
 * pages name the workload but not its output; the reading taken here makes it
 * the weighted counterpart of LayerNorm's reduce-then-reuse: per-column
 * weights w_j >= 0 (a second input vector),
 *   W = sum_j w_j,  mu = sum_j w_j x_j / W,
 *   var = sum_j w_j (x_j - mu)^2 / W,
 *   y_j = (x_j - mu) / sqrt(var + eps).
 * Rows with W == 0 are rejected.
 */
int oracle_weighted_std(const void *x, int dtype, int64_t rows, int64_t cols,
                        const void *w, int wdtype, double eps, double *y)
{
    int64_t r, j;
    if (!x || !w || !y || rows < 0 || cols <= 0 || !or_dtype_ok(dtype) ||
        !or_dtype_ok(wdtype) || !(eps >= 0.0))
        return OR_BAD_ARG;
    for (r = 0; r < rows; ++r) {
        int64_t base = r * cols;
        double W = 0.0, sw = 0.0, ssd = 0.0, mu, var, inv;
        for (j = 0; j < cols; ++j) {
            double wj = or_load(w, wdtype, j);
            if (!(wj >= 0.0))
                return OR_BAD_ARG;
            W += wj;
            sw += wj * or_load(x, dtype, base + j);
        }
        if (!(W > 0.0))
            return OR_BAD_ARG;
        mu = sw / W;
        for (j = 0; j < cols; ++j) {
            double d = or_load(x, dtype, base + j) - mu;
            ssd += or_load(w, wdtype, j) * d * d;
        }
        var = ssd / W;
        inv = 1.0 / sqrt(var + eps);
        for (j = 0; j < cols; ++j)
            y[base + j] = (or_load(x, dtype, base + j) - mu) * inv;
    }
    return OR_OK;
}

/*
 * Row-wise Pearson correlation of two matrices x and u of the same shape
 * (the Pearson workload of the CREDIT summary page, section "B. Workload-by-
 * Workload Scaling").  The pages name the workload only; the reading taken
 * here keeps the reduce-then-reuse shape: the statistics are the row means,
 * biased variances and covariance,
 *   mx = sum_j x_j / N,  mu = sum_j u_j / N,
 *   vx = sum_j (x_j - mx)^2 / N,  vu = sum_j (u_j - mu)^2 / N,
 *   cxu = sum_j (x_j - mx)(u_j - mu) / N,
 * and h writes every column's standardized co-deviation
 *   y_j = (x_j - mx)(u_j - mu) / sqrt((vx + eps)(vu + eps)),
 * whose row mean is the correlation r = cxu / sqrt((vx + eps)(vu + eps))
 * (Pearson's r when eps = 0), written to r[row].  Two passes per statistic,
 * every sum in fp64 in column order.  A row whose denominator is zero
 * (eps = 0 and a constant x or u) is rejected.
 */
int oracle_pearson(const void *x, const void *u, int dtype, int64_t rows, int64_t cols,
                   double eps, double *y, double *r)
{
    int64_t i, j;
    if (!x || !u || !y || !r || rows < 0 || cols <= 0 || !or_dtype_ok(dtype) || !(eps >= 0.0))
        return OR_BAD_ARG;
    for (i = 0; i < rows; ++i) {
        int64_t base = i * cols;
        double sx = 0.0, su = 0.0, mx, mu, sxx = 0.0, suu = 0.0, sxu = 0.0, den;
        for (j = 0; j < cols; ++j) {
            sx += or_load(x, dtype, base + j);
            su += or_load(u, dtype, base + j);
        }
        mx = sx / (double)cols;
        mu = su / (double)cols;
        for (j = 0; j < cols; ++j) {
            double dx = or_load(x, dtype, base + j) - mx;
            double du = or_load(u, dtype, base + j) - mu;
            sxx += dx * dx;
            suu += du * du;
            sxu += dx * du;
        }
        den = sqrt((sxx / (double)cols + eps) * (suu / (double)cols + eps));
        if (!(den > 0.0))
            return OR_BAD_ARG;
        for (j = 0; j < cols; ++j) {
            double dx = or_load(x, dtype, base + j) - mx;
            double du = or_load(u, dtype, base + j) - mu;
            y[base + j] = dx * du / den;
        }
        r[i] = (sxu / (double)cols) / den;
    }
    return OR_OK;
}
