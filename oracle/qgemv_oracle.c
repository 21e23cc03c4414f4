/*
 * qgemv_oracle.c -- plain, slow, fp64 CPU oracle for the dequant-fused
 * quantized matrix-vector product and its fused variants.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * source, header, table or helper with the CUDA path, and the CUDA path
 * never calls it.
 *
 * What it computes, and where the pages define it:
 *   - Weight format (planar, MLX style): 4-bit codes packed 8 per uint32,
 *     low nibble first along K; separate fp16 scale and bias tensors, one
 *     value per group of 64 consecutive k of a row.  "Boosting inference
 *     speed on Apple Silicon" (INFERENCE_RESEARCH.md), section 3, item 4
 *     (planar quantization, uint32-packed data, separate scales/biases,
 *     group 64).  2-bit codes (16 per uint32, low bits first) follow the
 *     same layout; the 2-bit experts are on the hada.io news page
 *     (topic 27758), "Resultats de performance" and "Shaders de calcul Metal".
 *     8-bit codes (4 per uint32, low byte first) likewise: Q8, the level the
 *     BaseRT page ("BaseRT: Best-in-Class LLM Inference on Apple Silicon via
 *     Native Metal") evaluates beside Q4.  oracle_code() reads any of the
 *     three widths (32 / bits codes per word).
 *   - Dequantisation w = q*scale + bias and its product with x: the hada.io
 *     page, "Noyau de dequantification optimise FMA" ((nibble*scale+bias)*x,
 *     rewritten as fma(nibble, scale*x, bias*x); an exact identity, so the
 *     oracle evaluates the plain product).
 *   - LUT / palettised 4-bit weights: the same 4-bit codes index a table
 *     of 16 fp16 values, w = lut[q]; INFERENCE_RESEARCH.md section 3,
 *     item 4 (add a LUT/palettised type: 4-bit indices plus a 16-entry
 *     f16 LUT, Core ML style).  One table serves rows_per_lut consecutive
 *     rows (all N: one table per tensor; 1: one per row).
 *   - Fusions RMSNorm->QKV, gate.up SwiGLU, MoE combine + residual:
 *     INFERENCE_RESEARCH.md section 1 (fusions to implement) and the hada.io
 *     page, "Shaders de calcul Metal" and "Deferred GPU Expert Compute".
 *
 * Every sum is taken in fp64 in index order; fp16 inputs convert to fp64
 * exactly; each fp16 output is rounded once, round-to-nearest-even.
 * Tolerance bounds (sum |w||x| etc.) are returned beside each result so
 * the tests can apply |y - y_ref| <= 2e-3 * bound + 1e-5.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_GROUP 64

/* ---------------------------------------------------------------- fp16 */

/* IEEE binary16 -> double.  Exact: every binary16 value is a double. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int mant = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);                 /* subnormal / zero */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25);  /* (1.m) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* double -> IEEE binary16, round to nearest, ties to even (one rounding). */
uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7E00;
    if (isinf(v))
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the value is an integer count of 2^-24 */
        double units = rint(ldexp(a, 24));            /* exact scaling; RNE */
        return sign | (uint16_t)units;                /* 1024 -> min normal */
    }
    int e;
    frexp(a, &e);                                     /* a in [2^(e-1), 2^e) */
    int E = e - 1;                                    /* unbiased exponent   */
    double m = rint(ldexp(a, 10 - E));                /* in [1024, 2048]     */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7C00;                         /* overflow -> inf */
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* ------------------------------------------------------------- unpack */

/* Number of uint32 words per row of K codes. */
static int64_t words_per_row(int bits, int K) { return (int64_t)K * bits / 32; }

/* Code q[n][k] of a packed row: codes are packed low bits first along K. */
int oracle_code(const uint32_t *row, int bits, int k)
{
    int per_word = 32 / bits;
    uint32_t word = row[k / per_word];
    int shift = bits * (k % per_word);
    return (int)((word >> shift) & ((1u << bits) - 1u));
}

/* Dequantised weight w[n][k] = q * scale[n][k/64] + bias[n][k/64], fp64. */
static double weight(const uint32_t *codes, const uint16_t *scales,
                     const uint16_t *biases, int bits, int K, int n, int k)
{
    int64_t G = K / ORACLE_GROUP;
    const uint32_t *row = codes + (int64_t)n * words_per_row(bits, K);
    int q = oracle_code(row, bits, k);
    double s = oracle_half_to_double(scales[(int64_t)n * G + k / ORACLE_GROUP]);
    double b = oracle_half_to_double(biases[(int64_t)n * G + k / ORACLE_GROUP]);
    return (double)q * s + b;
}

/* --------------------------------------------------------- threading */

static int g_threads = 0; /* 0 = OpenMP default */

void oracle_set_threads(int n) { g_threads = n; }

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------ dense matvec */

/*
 * y[n] = sum_k w[n][k] * x[k] for n in [0, N), x given in fp64.
 * absb[n] = sum_k |w[n][k]| * |x[k]| (nullable).  Rows are independent,
 * so they are split across threads; each row sums in index order.
 */
void oracle_matvec_f64(int bits, const uint32_t *codes, const uint16_t *scales,
                       const uint16_t *biases, int N, int K, const double *x,
                       double *y, double *absb)
{
    int nt = oracle_get_threads();
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int n = 0; n < N; ++n) {
        double acc = 0.0, mag = 0.0;
        for (int k = 0; k < K; ++k) {
            double w = weight(codes, scales, biases, bits, K, n, k);
            acc += w * x[k];
            mag += fabs(w) * fabs(x[k]);
        }
        y[n] = acc;
        if (absb)
            absb[n] = mag;
    }
}

/* out[n] = sum_k |w[n][k]| * v[k] for a non-negative fp64 vector v. */
static void abs_matvec(int bits, const uint32_t *codes, const uint16_t *scales,
                       const uint16_t *biases, int N, int K, const double *v,
                       double *out)
{
    int nt = oracle_get_threads();
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int n = 0; n < N; ++n) {
        double s = 0.0;
        for (int k = 0; k < K; ++k)
            s += fabs(weight(codes, scales, biases, bits, K, n, k)) * v[k];
        out[n] = s;
    }
}

/* ------------------------------------------------------- plain qgemv */

/*
 * qgemv: for each of M activation rows, y[m][n] = sum_k w[n][k] x[m][k]
 * (+ residual[m][n]).  y64 gets the fp64 value, y16 the fp16 rounding,
 * bound[m][n] = sum_k |w||x| + |residual| (the tolerance scale).
 * Any of y64, y16, bound may be NULL.
 */
void oracle_qgemv(int bits, const uint32_t *codes, const uint16_t *scales,
                  const uint16_t *biases, const uint16_t *x,
                  const uint16_t *residual, int M, int N, int K,
                  double *y64, uint16_t *y16, double *bound)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    double *yd = (double *)malloc(sizeof(double) * (size_t)N);
    double *ab = (double *)malloc(sizeof(double) * (size_t)N);
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < K; ++k)
            xd[k] = oracle_half_to_double(x[(int64_t)m * K + k]);
        oracle_matvec_f64(bits, codes, scales, biases, N, K, xd, yd, ab);
        for (int n = 0; n < N; ++n) {
            double v = yd[n], b = ab[n];
            if (residual) {
                double r = oracle_half_to_double(residual[(int64_t)m * N + n]);
                v += r;
                b += fabs(r);
            }
            int64_t o = (int64_t)m * N + n;
            if (y64) y64[o] = v;
            if (y16) y16[o] = oracle_double_to_half(v);
            if (bound) bound[o] = b;
        }
    }
    free(xd);
    free(yd);
    free(ab);
}

/* ------------------------------------------------ LUT / palettised */

/*
 * y[n] = sum_k lut[n / rows_per_lut][q[n][k]] * x[k] (+ residual[n]) for
 * 4-bit codes q (8 per uint32, low nibble first) and fp16 tables of 16
 * entries.  y64 = the fp64 value, y16 its fp16 rounding, bound = sum |w||x|
 * + |residual|.  Any of y64, y16, bound may be NULL.
 */
void oracle_lut_qgemv(const uint32_t *codes, const uint16_t *lut, int rows_per_lut,
                      const uint16_t *x, const uint16_t *residual, int N, int K,
                      double *y64, uint16_t *y16, double *bound)
{
    int nt = oracle_get_threads();
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int n = 0; n < N; ++n) {
        const uint32_t *row = codes + (int64_t)n * words_per_row(4, K);
        const uint16_t *table = lut + (int64_t)(n / rows_per_lut) * 16;
        double acc = 0.0, mag = 0.0;
        for (int k = 0; k < K; ++k) {
            double w = oracle_half_to_double(table[oracle_code(row, 4, k)]);
            double xv = oracle_half_to_double(x[k]);
            acc += w * xv;
            mag += fabs(w) * fabs(xv);
        }
        if (residual) {
            double r = oracle_half_to_double(residual[n]);
            acc += r;
            mag += fabs(r);
        }
        if (y64) y64[n] = acc;
        if (y16) y16[n] = oracle_double_to_half(acc);
        if (bound) bound[n] = mag;
    }
}

/* ----------------------------------------------------------- RMSNorm */

/* xn[k] = x[k] * gamma[k] / sqrt(mean(x^2) + eps); eps inside the root. */
void oracle_rmsnorm(const uint16_t *x, const uint16_t *gamma, int K, double eps,
                    double *xn)
{
    double ss = 0.0;
    for (int k = 0; k < K; ++k) {
        double v = oracle_half_to_double(x[k]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)K + eps);
    for (int k = 0; k < K; ++k)
        xn[k] = oracle_half_to_double(x[k]) * r * oracle_half_to_double(gamma[k]);
}

/* RMSNorm followed by the 4-bit matvec: y = W . rmsnorm(x). */
void oracle_rmsnorm_qgemv(const uint32_t *codes, const uint16_t *scales,
                          const uint16_t *biases, const uint16_t *x,
                          const uint16_t *gamma, double eps, int N, int K,
                          double *y64, uint16_t *y16, double *bound)
{
    double *xn = (double *)malloc(sizeof(double) * (size_t)K);
    double *yd = (double *)malloc(sizeof(double) * (size_t)N);
    double *ab = (double *)malloc(sizeof(double) * (size_t)N);
    oracle_rmsnorm(x, gamma, K, eps, xn);
    oracle_matvec_f64(4, codes, scales, biases, N, K, xn, yd, ab);
    for (int n = 0; n < N; ++n) {
        if (y64) y64[n] = yd[n];
        if (y16) y16[n] = oracle_double_to_half(yd[n]);
        if (bound) bound[n] = ab[n];
    }
    free(xn);
    free(yd);
    free(ab);
}

/* ------------------------------------------------------------ SwiGLU */

/* silu(z) = z / (1 + e^-z), in fp64. */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Gate.up SwiGLU on an fp64 input xt: g = Wg xt, u = Wu xt,
 * h = silu(g) * u.  tol[i] is the first-order error budget of h[i]:
 *   dg = 2e-3 sum|Wg||xt|, du = 2e-3 sum|Wu||xt|,
 *   tol = 1.1 |u| dg + |silu(g)| du + 2^-11 |h| + 1e-5
 * (1.1 bounds |silu'|; 2^-11 |h| is one fp16 rounding of h).
 */
static void swiglu_core(const uint32_t *gc, const uint16_t *gs, const uint16_t *gb,
                        const uint32_t *uc, const uint16_t *us, const uint16_t *ub,
                        const double *xt, int I, int K, double *h, double *tol)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *ag = (double *)malloc(sizeof(double) * (size_t)I);
    double *au = (double *)malloc(sizeof(double) * (size_t)I);
    oracle_matvec_f64(4, gc, gs, gb, I, K, xt, g, ag);
    oracle_matvec_f64(4, uc, us, ub, I, K, xt, u, au);
    for (int i = 0; i < I; ++i) {
        double sg = oracle_silu(g[i]);
        h[i] = sg * u[i];
        if (tol)
            tol[i] = 1.1 * fabs(u[i]) * (2e-3 * ag[i]) + fabs(sg) * (2e-3 * au[i]) +
                     ldexp(fabs(h[i]), -11) + 1e-5;
    }
    free(g);
    free(u);
    free(ag);
    free(au);
}

/*
 * swiglu_qgemv: h[i] = silu(Wg[i] . xt) * (Wu[i] . xt) with xt = x, or
 * xt = rmsnorm(x) when gamma is given (the fused post-attention norm).
 */
void oracle_swiglu_qgemv(const uint32_t *gc, const uint16_t *gs, const uint16_t *gb,
                         const uint32_t *uc, const uint16_t *us, const uint16_t *ub,
                         const uint16_t *x, const uint16_t *gamma, double eps,
                         int I, int K, double *h64, uint16_t *h16, double *tol)
{
    double *xt = (double *)malloc(sizeof(double) * (size_t)K);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    if (gamma)
        oracle_rmsnorm(x, gamma, K, eps, xt);
    else
        for (int k = 0; k < K; ++k)
            xt[k] = oracle_half_to_double(x[k]);
    swiglu_core(gc, gs, gb, uc, us, ub, xt, I, K, h, tol);
    for (int i = 0; i < I; ++i) {
        if (h64) h64[i] = h[i];
        if (h16) h16[i] = oracle_double_to_half(h[i]);
    }
    free(xt);
    free(h);
}

/* --------------------------------------------------------------- MoE */

/*
 * MoE top-K expert matvec with weighted combine and residual:
 *   for each k < top_k: e = idx[k]; if e is outside [0, E) set *err = 1
 *   and drop that expert; else h_k = swiglu(Wgu[e] gate rows 0..I-1,
 *   up rows I..2I-1, x) in fp64 (unrounded), and
 *   y[n] = r[n] + sum_k wt[k] * (Wd[e] h_k)[n], rounded once to fp16.
 * Experts are stored contiguously: gate.up [E][2I][K/8] words with
 * [E][2I][H/64] scales/biases (K = H), down [E][H][I/8] words with
 * [E][H][I/64] scales/biases.
 * tol[n] = 2e-3 (sum_k wt_k sum_j |Wd_nj| (|h_kj| + tol_h_kj / 2e-3) + |r_n|) + 1e-5.
 * A repeated expert index counts as two contributions.
 */
void oracle_moe_qgemv_combine(const uint32_t *gu_codes, const uint16_t *gu_scales,
                              const uint16_t *gu_biases, const uint32_t *dn_codes,
                              const uint16_t *dn_scales, const uint16_t *dn_biases,
                              int n_experts, int H, int I, const int32_t *idx,
                              const float *wt, int top_k, const uint16_t *x,
                              const uint16_t *residual, double *y64, uint16_t *y16,
                              double *tol, int *err)
{
    int64_t gu_words = (int64_t)2 * I * words_per_row(4, H);
    int64_t gu_groups = (int64_t)2 * I * (H / ORACLE_GROUP);
    int64_t dn_words = (int64_t)H * words_per_row(4, I);
    int64_t dn_groups = (int64_t)H * (I / ORACLE_GROUP);
    double *xt = (double *)malloc(sizeof(double) * (size_t)H);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    double *th = (double *)malloc(sizeof(double) * (size_t)I);
    double *hb = (double *)malloc(sizeof(double) * (size_t)I);
    double *yd = (double *)malloc(sizeof(double) * (size_t)H);
    double *ab = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)calloc((size_t)H, sizeof(double));
    double *mag = (double *)calloc((size_t)H, sizeof(double));
    if (err)
        *err = 0;
    for (int k = 0; k < H; ++k)
        xt[k] = oracle_half_to_double(x[k]);
    for (int t = 0; t < top_k; ++t) {
        int e = idx[t];
        if (e < 0 || e >= n_experts) {
            if (err)
                *err = 1;
            continue;
        }
        const uint32_t *gc = gu_codes + (int64_t)e * gu_words;
        const uint16_t *gs = gu_scales + (int64_t)e * gu_groups;
        const uint16_t *gb = gu_biases + (int64_t)e * gu_groups;
        int64_t up_w = (int64_t)I * words_per_row(4, H);
        int64_t up_g = (int64_t)I * (H / ORACLE_GROUP);
        swiglu_core(gc, gs, gb, gc + up_w, gs + up_g, gb + up_g, xt, I, H, h, th);
        /* y contribution, and its error bound through |Wd| (|h| + tol_h / 2e-3) */
        for (int j = 0; j < I; ++j)
            hb[j] = fabs(h[j]) + th[j] / 2e-3;
        const uint32_t *dc = dn_codes + (int64_t)e * dn_words;
        const uint16_t *ds = dn_scales + (int64_t)e * dn_groups;
        const uint16_t *db = dn_biases + (int64_t)e * dn_groups;
        oracle_matvec_f64(4, dc, ds, db, H, I, h, yd, NULL);
        abs_matvec(4, dc, ds, db, H, I, hb, ab);
        double w = (double)wt[t];
        for (int n = 0; n < H; ++n)
            acc[n] += w * yd[n];
        for (int n = 0; n < H; ++n)
            mag[n] += fabs(w) * ab[n];
    }
    for (int n = 0; n < H; ++n) {
        double r = residual ? oracle_half_to_double(residual[n]) : 0.0;
        double v = acc[n] + r;
        if (y64) y64[n] = v;
        if (y16) y16[n] = oracle_double_to_half(v);
        if (tol) tol[n] = 2e-3 * (mag[n] + fabs(r)) + 1e-5;
    }
    free(xt);
    free(h);
    free(th);
    free(hb);
    free(yd);
    free(ab);
    free(acc);
    free(mag);
}
