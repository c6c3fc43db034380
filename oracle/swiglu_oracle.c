/*
 * swiglu_oracle.c -- plain, slow, obviously-correct CPU oracle for the SwiGLU
 * MLP block (forward and the full backward chain).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library; it reads the same bf16 input bits and works in fp64.
 *
 * What it computes (notation of the "SwiGLU MLP Drop-H technical report",
 * lgystoic.github.io/notes/swiglu-mlp-drop-h/, section "original math of the
 * SwiGLU MLP", forward and backward formulas):
 *
 *   preact = x @ W1^T               x [M,D], W1 [2H,D]   -> preact [M,2H]
 *   left, gate = split(preact)      left = columns [0,H), gate = [H,2H)
 *   h      = left * silu(gate)      silu(g) = g * sigma(g)
 *   y      = h @ W2^T               W2 [Dout,H]          -> y [M,Dout]
 *
 *   grad_h      = dy @ W2           dy [M,Dout]          -> [M,H]
 *   dleft       = grad_h * silu(gate)
 *   dgate       = grad_h * left * silu'(gate)
 *   grad_preact = [dleft | dgate]                        -> [M,2H]
 *   dx          = grad_preact @ W1                       -> [M,D]
 *   dW1         = grad_preact^T @ x   (one merged [2H,M]@[M,D] product)
 *   dW2         = dy^T @ h                               -> [Dout,H]
 *
 * silu'(g) is taken in the form sigma(g) * (1 + g * (1 - sigma(g))), one of
 * the three equal forms listed in the "SwiGLU MLP forward/backward
 * optimization" note (lgystoic.github.io/notes/
 * swiglu-mlp-forward-backward-optimization/), section 2 "Backward".
 *
 * Rounding (round_mode = 1): the tensors the method keeps in HBM as bf16 are
 * rounded to bf16 (round-to-nearest-even) at exactly the point they are
 * stored: preact, h and grad_preact.  h follows the drop-h report's fused
 * backward kernel pseudo-code, h = bf16(left) * bf16(silu): silu is rounded
 * to bf16 before the product and the product is rounded once more when it is
 * stored.  grad_h is never rounded (the fused path never stores it).  The
 * final outputs y, dx, dW1, dW2 are returned unrounded in fp64.
 * round_mode = 0 keeps every intermediate in exact fp64 (used by the
 * finite-difference and autograd pins).
 *
 * residual = 1 gives the residual block y = x + MLP(x) (requires D == Dout), the
 * "Residual Add Epilogue" of the lesson "Transformer MLP, GEMM and operator fusion"
 * (lincklin.cn, section 24: the down projection's output plus the block input); its
 * backward adds dy to dx (the identity path), the weight gradients are unchanged.
 *
 * Every loop is a plain sum over the contraction index in ascending order;
 * OpenMP only splits independent output rows/columns across threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE fp32). */
static double bf16_bits_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* An input matrix: bf16 bit patterns (f64 == 0) or fp64 values (f64 == 1).
 * The fp64 form lets the finite-difference pins perturb inputs by amounts no
 * bf16 value can carry. */
typedef struct { const void *p; int f64; } oracle_mat;

static double at(oracle_mat a, int64_t i) {
    return a.f64 ? ((const double *)a.p)[i] : bf16_bits_to_f64(((const uint16_t *)a.p)[i]);
}

/* Largest finite bf16: (2 - 2^-7) * 2^127. */
#define ORACLE_BF16_MAX 3.3895313892515355e38

/* Round a double to the nearest bf16 value, ties to even, returned as a
 * double.  bf16 keeps 8 significant bits and fp32's exponent range
 * (normal down to 2^-126, subnormal quantum 2^-133). */
double oracle_round_bf16(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    frexp(v, &e);           /* v = f * 2^e with 0.5 <= |f| < 1 */
    int q = e - 8;          /* exponent of one unit in the last place */
    if (q < -133) q = -133;
    double r = ldexp(nearbyint(ldexp(v, -q)), q);   /* default mode: ties-to-even */
    if (fabs(r) > ORACLE_BF16_MAX) r = copysign(INFINITY, v);
    return r;
}

/* Logistic sigmoid, silu and its derivative, straight from the definitions. */
double oracle_sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }
double oracle_silu(double g) { return g * oracle_sigmoid(g); }
double oracle_silu_prime(double g) {
    double s = oracle_sigmoid(g);
    return s * (1.0 + g * (1.0 - s));
}

static double maybe_round(double v, int round_mode) {
    return round_mode ? oracle_round_bf16(v) : v;
}

/* h from one (left, gate) pair, as stored by the method. */
static double swiglu_h(double left, double gate, int round_mode) {
    return maybe_round(left * maybe_round(oracle_silu(gate), round_mode), round_mode);
}

static double *to_f64(oracle_mat src, int64_t n) {
    double *dst = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!dst) return NULL;
    for (int64_t i = 0; i < n; ++i) dst[i] = at(src, i);
    return dst;
}

/*
 * Forward pass for a subset of token rows.
 *   in_f64: 0 = every input is bf16 bit patterns, 1 = every input is fp64.
 *   rows[nrows]: row indices into x (rows == NULL means rows 0..nrows-1).
 *   Outputs are dense [nrows, *] fp64 arrays; any may be NULL:
 *     preact_out [nrows, 2H]  (bf16-rounded when round_mode = 1)
 *     h_out      [nrows, H]   (bf16-rounded when round_mode = 1)
 *     y_out      [nrows, Dout] (unrounded)
 * Returns 0 on success, -1 on allocation failure.
 */
int oracle_swiglu_fwd(const void *x_p, const void *W1_p, const void *W2_p, int in_f64,
                      int64_t M, int64_t D, int64_t H, int64_t Dout,
                      const int64_t *rows, int64_t nrows, int round_mode, int residual,
                      double *preact_out, double *h_out, double *y_out) {
    (void)M;
    oracle_mat x = {x_p, in_f64};
    double *w1 = to_f64((oracle_mat){W1_p, in_f64}, 2 * H * D);
    double *w2 = to_f64((oracle_mat){W2_p, in_f64}, Dout * H);
    if (!w1 || !w2) { free(w1); free(w2); return -1; }
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        double *xr = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
        double *pre = (double *)malloc((size_t)(2 * H > 0 ? 2 * H : 1) * sizeof(double));
        double *hr = (double *)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
        if (!xr || !pre || !hr) {
            free(xr); free(pre); free(hr);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        for (int64_t d = 0; d < D; ++d) xr[d] = at(x, m * D + d);
        /* preact[m, n] = sum_d x[m, d] * W1[n, d] */
        for (int64_t n = 0; n < 2 * H; ++n) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += xr[d] * w1[n * D + d];
            pre[n] = maybe_round(acc, round_mode);
        }
        /* h[m, j] = left * silu(gate), left = preact[m, j], gate = preact[m, H + j] */
        for (int64_t j = 0; j < H; ++j) hr[j] = swiglu_h(pre[j], pre[H + j], round_mode);
        /* y[m, o] = sum_j h[m, j] * W2[o, j] */
        if (y_out) {
            for (int64_t o = 0; o < Dout; ++o) {
                double acc = 0.0;
                for (int64_t j = 0; j < H; ++j) acc += hr[j] * w2[o * H + j];
                /* residual block: y = x + MLP(x) (needs D == Dout) */
                y_out[i * Dout + o] = residual ? xr[o] + acc : acc;
            }
        }
        if (preact_out) memcpy(preact_out + i * 2 * H, pre, (size_t)(2 * H) * sizeof(double));
        if (h_out) memcpy(h_out + i * H, hr, (size_t)H * sizeof(double));
        free(xr); free(pre); free(hr);
    }
    free(w1); free(w2);
    return fail ? -1 : 0;
}

/*
 * Backward pass, row-wise outputs, for a subset of token rows.  Inputs are the
 * saved preact [M,2H] and the upstream gradient dy [M,Dout].
 *   grad_h_out      [nrows, H]   grad_h = dy @ W2 (never rounded)
 *   grad_preact_out [nrows, 2H]  [dleft | dgate] (rounded when round_mode = 1)
 *   h_out           [nrows, H]   h recomputed from preact (rounded likewise)
 *   dx_out          [nrows, D]   dx = grad_preact @ W1 (unrounded)
 * Any output pointer may be NULL.
 */
int oracle_swiglu_bwd_rows(const void *W1_p, const void *W2_p,
                           const void *preact_p, const void *dy_p, int in_f64,
                           int64_t M, int64_t D, int64_t H, int64_t Dout,
                           const int64_t *rows, int64_t nrows, int round_mode, int residual,
                           double *grad_h_out, double *grad_preact_out,
                           double *h_out, double *dx_out) {
    (void)M;
    oracle_mat preact = {preact_p, in_f64}, dy = {dy_p, in_f64};
    double *w1 = to_f64((oracle_mat){W1_p, in_f64}, 2 * H * D);
    double *w2 = to_f64((oracle_mat){W2_p, in_f64}, Dout * H);
    if (!w1 || !w2) { free(w1); free(w2); return -1; }
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        double *gh = (double *)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
        double *gp = (double *)malloc((size_t)(2 * H > 0 ? 2 * H : 1) * sizeof(double));
        double *dxr = (double *)calloc((size_t)(D > 0 ? D : 1), sizeof(double));
        if (!gh || !gp || !dxr) {
            free(gh); free(gp); free(dxr);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        /* grad_h[m, j] = sum_o dy[m, o] * W2[o, j]   (o ascending for every j) */
        for (int64_t o = 0; o < Dout; ++o) {
            double g = at(dy, m * Dout + o);
            const double *w2r = w2 + o * H;
            for (int64_t j = 0; j < H; ++j) gh[j] += g * w2r[j];
        }
        for (int64_t j = 0; j < H; ++j) {
            double left = at(preact, m * 2 * H + j);
            double gate = at(preact, m * 2 * H + H + j);
            double dleft = gh[j] * oracle_silu(gate);
            double dgate = gh[j] * left * oracle_silu_prime(gate);
            gp[j] = maybe_round(dleft, round_mode);
            gp[H + j] = maybe_round(dgate, round_mode);
            if (h_out) h_out[i * H + j] = swiglu_h(left, gate, round_mode);
        }
        /* dx[m, d] = sum_r grad_preact[m, r] * W1[r, d]   (r ascending for every d) */
        for (int64_t r = 0; r < 2 * H; ++r) {
            double g = gp[r];
            const double *w1r = w1 + r * D;
            for (int64_t d = 0; d < D; ++d) dxr[d] += g * w1r[d];
        }
        /* residual block: the identity path adds dy to dx (needs D == Dout) */
        if (residual)
            for (int64_t d = 0; d < D; ++d) dxr[d] += at(dy, m * Dout + d);
        if (grad_h_out) memcpy(grad_h_out + i * H, gh, (size_t)H * sizeof(double));
        if (grad_preact_out) memcpy(grad_preact_out + i * 2 * H, gp, (size_t)(2 * H) * sizeof(double));
        if (dx_out) memcpy(dx_out + i * D, dxr, (size_t)D * sizeof(double));
        free(gh); free(gp); free(dxr);
    }
    free(w1); free(w2);
    return fail ? -1 : 0;
}

/*
 * Backward pass, weight gradients, for a subset of hidden indices j.
 * For every selected j (cols[k] = j, cols == NULL means j = k):
 *   dW2_out  [ncols, Dout] : row k holds the column dW2[:, j] = sum_m dy[m,:] * h[m, j]
 *   dW1_out  [2*ncols, D]  : row k holds dW1[j, :]         = sum_m dleft[m, j] * x[m, :]
 *                            row ncols+k holds dW1[H+j, :] = sum_m dgate[m, j] * x[m, :]
 * h, dleft and dgate are recomputed for all M rows from preact and dy with the
 * same formulas (and roundings) as oracle_swiglu_bwd_rows.  Sums run over m
 * ascending.
 */
int oracle_swiglu_bwd_cols(const void *x_p, const void *W2_p,
                           const void *preact_p, const void *dy_p, int in_f64,
                           int64_t M, int64_t D, int64_t H, int64_t Dout,
                           const int64_t *cols, int64_t ncols, int round_mode,
                           double *dW2_out, double *dW1_out) {
    oracle_mat x = {x_p, in_f64}, W2 = {W2_p, in_f64};
    oracle_mat preact = {preact_p, in_f64}, dy = {dy_p, in_f64};
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t k = 0; k < ncols; ++k) {
        int64_t j = cols ? cols[k] : k;
        int64_t na = (Dout > D ? Dout : D);
        double *w2c = (double *)malloc((size_t)(Dout > 0 ? Dout : 1) * sizeof(double));
        double *hcol = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
        double *dl = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
        double *dg = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
        double *acc = (double *)malloc((size_t)(na > 0 ? na : 1) * sizeof(double));
        if (!w2c || !hcol || !dl || !dg || !acc) {
            free(w2c); free(hcol); free(dl); free(dg); free(acc);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        for (int64_t o = 0; o < Dout; ++o) w2c[o] = at(W2, o * H + j);
        for (int64_t m = 0; m < M; ++m) {
            double gh = 0.0;   /* grad_h[m, j] = sum_o dy[m, o] * W2[o, j] */
            for (int64_t o = 0; o < Dout; ++o) gh += at(dy, m * Dout + o) * w2c[o];
            double left = at(preact, m * 2 * H + j);
            double gate = at(preact, m * 2 * H + H + j);
            hcol[m] = swiglu_h(left, gate, round_mode);
            dl[m] = maybe_round(gh * oracle_silu(gate), round_mode);
            dg[m] = maybe_round(gh * left * oracle_silu_prime(gate), round_mode);
        }
        if (dW2_out) {
            for (int64_t o = 0; o < Dout; ++o) acc[o] = 0.0;
            for (int64_t m = 0; m < M; ++m)
                for (int64_t o = 0; o < Dout; ++o) acc[o] += at(dy, m * Dout + o) * hcol[m];
            memcpy(dW2_out + k * Dout, acc, (size_t)Dout * sizeof(double));
        }
        if (dW1_out) {
            for (int half = 0; half < 2; ++half) {
                const double *g = half ? dg : dl;
                for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
                for (int64_t m = 0; m < M; ++m)
                    for (int64_t d = 0; d < D; ++d) acc[d] += g[m] * at(x, m * D + d);
                memcpy(dW1_out + (half * ncols + k) * D, acc, (size_t)D * sizeof(double));
            }
        }
        free(w2c); free(hcol); free(dl); free(dg); free(acc);
    }
    return fail ? -1 : 0;
}

/* Threads the OpenMP runtime will use (reported as the baseline's core count). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * FP8 forward with a quantising epilogue.
 *
 * "Lesson 24: MLP, GEMM and operator fusion in the Transformer" (lincklin.cn),
 * section 26 (quantised GEMM epilogue): the 8-bit GEMM accumulates in higher
 * precision and the epilogue scales the accumulator, applies the activation,
 * rounds and saturates to the 8-bit output format, y = sat8(round(s * acc + b));
 * section 31: 8-bit weights halve the weight traffic of the bandwidth-bound
 * decode step.
 *
 * The 8-bit format is FP8 E4M3 ("e4m3fn": 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent field 0 is subnormal, (m / 8) * 2^-6; the code
 * with all exponent and mantissa bits set is NaN; no infinities; the largest
 * finite value is 1.75 * 2^8 = 448).
 *
 * The block in FP8 (per-tensor scales; the block has no bias, b = 0):
 *   x = s_x * x8,  W1 = s_w1 * W1_8,  W2 = s_w2 * W2_8        (8-bit codes)
 *   preact = s_x * s_w1 * (x8 @ W1_8^T)          accumulated exactly, stored bf16
 *   h      = left * bf16(silu(gate))             from the bf16 preact, as in fp64
 *   h8     = sat8(round(h / s_h))                the quantising epilogue
 *   y      = s_h * s_w2 * (h8 @ W2_8^T)          returned unrounded
 * Products of two E4M3 values are exact in fp64 and so are sums of up to 2^20 of
 * them (their exponents span fewer than 36 bits), so both accumulations are
 * exact here in any order.
 * ------------------------------------------------------------------------ */

double oracle_e4m3_decode(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);   /* (m/8) 2^-6 | (1 + m/8) 2^(e-7) */
    return s ? -v : v;
}

/* Nearest E4M3 code, ties to the even code (mantissa LSB 0); magnitudes beyond
 * 448 saturate to +-448; NaN gives the NaN code. */
int oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    int sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 0x7F; ++c) {       /* all non-negative finite codes, ascending */
        double err = fabs(oracle_e4m3_decode(c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return sign | best;                    /* beyond 448 the nearest code is 448 itself */
}

int oracle_swiglu_fwd_fp8(const uint8_t *x8, const uint8_t *W1_8, const uint8_t *W2_8,
                          double s_x, double s_w1, double s_w2, double s_h,
                          int64_t M, int64_t D, int64_t H, int64_t Dout,
                          const int64_t *rows, int64_t nrows,
                          double *preact_out, double *hpre_out, uint8_t *h8_out, double *y_out) {
    (void)M;
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = oracle_e4m3_decode(c);
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        double *pre = (double *)malloc((size_t)(2 * H > 0 ? 2 * H : 1) * sizeof(double));
        double *hq = (double *)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
        if (!pre || !hq) {
            free(pre); free(hq);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        for (int64_t n = 0; n < 2 * H; ++n) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += lut[x8[m * D + d]] * lut[W1_8[n * D + d]];
            pre[n] = oracle_round_bf16(s_x * s_w1 * acc);
        }
        for (int64_t j = 0; j < H; ++j) {
            double h = pre[j] * oracle_round_bf16(oracle_silu(pre[H + j]));
            int code = oracle_e4m3_encode(h / s_h);
            if (hpre_out) hpre_out[i * H + j] = h;
            if (h8_out) h8_out[i * H + j] = (uint8_t)code;
            hq[j] = lut[code];
        }
        if (y_out) {
            for (int64_t o = 0; o < Dout; ++o) {
                double acc = 0.0;
                for (int64_t j = 0; j < H; ++j) acc += hq[j] * lut[W2_8[o * H + j]];
                y_out[i * Dout + o] = s_h * s_w2 * acc;
            }
        }
        if (preact_out) memcpy(preact_out + i * 2 * H, pre, (size_t)(2 * H) * sizeof(double));
        free(pre); free(hq);
    }
    return fail ? -1 : 0;
}
