/*
 * tcq_oracle.c -- plain CPU oracle for the packed trellis-coded weight matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (libtrellis, its
 * Python binding) may include, link or call this file.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * The oracle follows the plain definition of what the method computes, step
 * by step and in double precision where the pages leave precision open:
 *
 *   1. block bitstring   S[j] = bit (j mod 32) of word floor(j/32), j < BT*k
 *   2. window            win(t) = sum_{i<L} S[(p+i) mod BT*k] 2^i,
 *                        p = (BT-1-t)*k           (tail-biting wrap)
 *   3. weight            w = bf16_rne( f32( lut[win] * f32(scale[row]) ) )
 *   4. contraction       axis 1: y[m][r] = sum_c x[m][c] w[r][c]
 *                        axis 0: y[m][c] = sum_r x[m][r] w[r][c]
 *                        accumulated in double
 *   5. output            out = bf16_rne(y), rounded directly from double
 *
 * Sources (the pages):
 *   - @mlx-bun/inference 1.0.0, kernels/trellis/tiled-prefill.ts, prefill tile
 *     kernel: block word addressing, window position (BT-1-t)*k, word-local
 *     shift, the spill into the next word that wraps to word 0 of the block,
 *     the L-bit mask, the weight T(value*scale), fp32 accumulation and the
 *     rounding of the output to T.
 *   - @mlx-bun/inference 1.0.0, kernels/trellis/vector-expand.ts, expand
 *     kernel: the interleave-2 block layout, and "earlier weights occupy the
 *     higher bits" of a shared window.
 *   - @mlx-bun/inference 1.0.0, kernels/trellis/scatter.ts, scatter kernels
 *     and launch: axis-0 index map, split ranges rowsPer = ceil(R/SPLITS),
 *     fp32 partials [M, SPLITS, C] and their sum over the split axis.
 *   - the codebook value is an explicit f32 table lut[2^L] (the codebook
 *     module is not on the pages; the expansion is said to consume the
 *     precise host LUT).
 *
 * Every rounding here is written from the IEEE 754 definition of round to
 * nearest, ties to even.  No function of this file is tuned for speed.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#include <fenv.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* threads                                                                  */
/* ------------------------------------------------------------------------ */

void tcq_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int tcq_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bfloat16                                                                 */
/* ------------------------------------------------------------------------ */

/* bf16 -> float: a bf16 is the upper half of an IEEE binary32 pattern. */
float tcq_oracle_bf16_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round a real value (given exactly as a double) to the nearest bf16 value,
 * ties to the value with an even last mantissa bit.  bf16 keeps 7 stored
 * fraction bits and the binary32 exponent range; below 2^-126 its spacing is
 * the subnormal quantum 2^-133.  The quantum of the binade of |y| is found,
 * |y| is divided by it (exact: a power of two), rounded to the nearest
 * integer with ties to even (nearbyint in the default rounding mode) and
 * scaled back.  A result of 2^128 or more is an overflow to infinity.
 */
uint16_t tcq_oracle_bf16_from_double(double y) {
    uint16_t sign = signbit(y) ? 0x8000u : 0x0000u;
    if (isnan(y)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(y)) return (uint16_t)(sign | 0x7F80u);
    double a = fabs(y);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);            /* 2^(e-1) <= a < 2^e */
    int q = (e - 1) - 7;           /* spacing of bf16 values in [2^(e-1), 2^e) */
    if (q < -133) q = -133;        /* subnormal range */
    double r = ldexp(a, -q);
    if (fegetround() != FE_TONEAREST) fesetround(FE_TONEAREST);
    double n = nearbyint(r);       /* nearest integer, ties to even */
    double v = ldexp(n, q);        /* the rounded magnitude, a bf16 value */
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;            /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* float -> bf16: the float is exactly a double, so one rounding. */
uint16_t tcq_oracle_bf16_from_float(float f) {
    return tcq_oracle_bf16_from_double((double)f);
}

/* Vector forms for the Python wrapper. */
void tcq_oracle_bf16_from_double_n(const double* y, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = tcq_oracle_bf16_from_double(y[i]);
}
void tcq_oracle_bf16_from_float_n(const float* y, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = tcq_oracle_bf16_from_float(y[i]);
}

/* ------------------------------------------------------------------------ */
/* geometry                                                                 */
/* ------------------------------------------------------------------------ */

/* words of one block: BT symbols of k bits, packed into 32-bit words */
static int64_t words_per_block(int bt, int k) { return (int64_t)bt * k / 32; }

/*
 * First word of block b of row r.
 *   interleave 0: rows are contiguous, blocks contiguous inside a row.
 *   interleave 2: pairs of blocks of all rows are grouped: base =
 *                 (b/2)*R*2*wpb + r*2*wpb + (b%2)*wpb.
 */
static int64_t block_base(int64_t r, int64_t b, int64_t rows, int64_t cols,
                          int bt, int k, int interleave) {
    int64_t wpb = words_per_block(bt, k);
    if (interleave == 2)
        return (b / 2) * rows * 2 * wpb + r * 2 * wpb + (b % 2) * wpb;
    return r * (cols / bt) * wpb + b * wpb;
}

/* ------------------------------------------------------------------------ */
/* windows                                                                  */
/* ------------------------------------------------------------------------ */

/* bit j of the block bitstring: least significant bit of word 0 first */
static uint32_t block_bit(const uint32_t* words, int64_t j) {
    return (words[j / 32] >> (j % 32)) & 1u;
}

/* L-bit window of column t of one block, taken bit by bit, circularly. */
uint32_t tcq_oracle_window(const uint32_t* block_words, int bt, int k, int L, int t) {
    int64_t n = (int64_t)bt * k;
    int64_t p = (int64_t)(bt - 1 - t) * k;
    uint32_t v = 0;
    for (int i = 0; i < L; i++)
        v |= block_bit(block_words, (p + i) % n) << i;
    return v;
}

/* decoded weight w[r][c] (bf16 bits), with its window */
static uint16_t weight_at(const uint32_t* codes, int64_t rows, int64_t cols,
                          int bt, int k, int L, int interleave,
                          const uint16_t* scales, const float* lut,
                          int64_t r, int64_t c, uint32_t* win_out) {
    int64_t b = c / bt;
    int t = (int)(c % bt);
    const uint32_t* bw = codes + block_base(r, b, rows, cols, bt, k, interleave);
    uint32_t win = tcq_oracle_window(bw, bt, k, L, t);
    if (win_out) *win_out = win;
    float value = lut[win];
    float s = tcq_oracle_bf16_to_float(scales[r]);
    /* f32(value * s): the exact product (24 x 8 significant bits fits a
       double) rounded once to binary32 */
    float prod = (float)((double)value * (double)s);
    return tcq_oracle_bf16_from_float(prod);
}

uint16_t tcq_oracle_weight(const uint32_t* codes, int64_t rows, int64_t cols,
                           int bt, int k, int L, int interleave,
                           const uint16_t* scales, const float* lut,
                           int64_t r, int64_t c) {
    return weight_at(codes, rows, cols, bt, k, L, interleave, scales, lut, r, c, NULL);
}

/*
 * Expand the whole matrix: w_out bf16 [rows, cols], win_out u16 [rows, cols]
 * (either may be NULL).
 */
void tcq_oracle_expand(const uint32_t* codes, int64_t rows, int64_t cols,
                       int bt, int k, int L, int interleave,
                       const uint16_t* scales, const float* lut,
                       uint16_t* w_out, uint16_t* win_out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) {
            uint32_t win;
            uint16_t w = weight_at(codes, rows, cols, bt, k, L, interleave,
                                   scales, lut, r, c, &win);
            if (w_out) w_out[r * cols + c] = w;
            if (win_out) win_out[r * cols + c] = (uint16_t)win;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* contractions on expanded weights                                          */
/* ------------------------------------------------------------------------ */

/*
 * Axis 1 (rows are output features): x bf16 [M, cols], w bf16 [rows, cols].
 * y[m][r] = sum_c x[m][c] w[r][c] and a[m][r] = sum_c |x[m][c] w[r][c]|,
 * both double [M, rows]; out bf16 [M, rows].  Any output may be NULL.
 */
void tcq_oracle_matmul_axis1(const uint16_t* x, int64_t M, const uint16_t* w,
                             int64_t rows, int64_t cols,
                             double* y, double* a, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, sa = 0.0;
            for (int64_t c = 0; c < cols; c++) {
                double p = (double)tcq_oracle_bf16_to_float(x[m * cols + c]) *
                           (double)tcq_oracle_bf16_to_float(w[r * cols + c]);
                s += p;
                sa += fabs(p);
            }
            if (y) y[m * rows + r] = s;
            if (a) a[m * rows + r] = sa;
            if (out) out[m * rows + r] = tcq_oracle_bf16_from_double(s);
        }
    }
}

/*
 * Axis 0 (rows are input features): x bf16 [M, rows], w bf16 [rows, cols].
 * y[m][c] = sum_r x[m][r] w[r][c].  With splits > 0 the row range is cut into
 * splits ranges of rp = ceil(rows/splits) rows, split s covering
 * [s*rp, min(rows, (s+1)*rp)) (empty past the end), and partial[m][s][c]
 * (double [M, splits, cols]) holds each range's sum.  y is the sum over all
 * rows taken in row order.
 */
void tcq_oracle_matmul_axis0(const uint16_t* x, int64_t M, const uint16_t* w,
                             int64_t rows, int64_t cols, int64_t splits,
                             double* y, double* a, uint16_t* out, double* partial) {
    int64_t rp = splits > 0 ? (rows + splits - 1) / splits : rows;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; c++) {
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, sa = 0.0;
            for (int64_t r = 0; r < rows; r++) {
                double p = (double)tcq_oracle_bf16_to_float(x[m * rows + r]) *
                           (double)tcq_oracle_bf16_to_float(w[r * cols + c]);
                s += p;
                sa += fabs(p);
            }
            if (y) y[m * cols + c] = s;
            if (a) a[m * cols + c] = sa;
            if (out) out[m * cols + c] = tcq_oracle_bf16_from_double(s);
            if (partial && splits > 0) {
                for (int64_t sp = 0; sp < splits; sp++) {
                    int64_t r0 = sp * rp, r1 = r0 + rp < rows ? r0 + rp : rows;
                    double ps = 0.0;
                    for (int64_t r = r0; r < r1; r++)
                        ps += (double)tcq_oracle_bf16_to_float(x[m * rows + r]) *
                              (double)tcq_oracle_bf16_to_float(w[r * cols + c]);
                    partial[(m * splits + sp) * cols + c] = ps;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* sampled outputs straight from the codes (for matrices too big to expand)  */
/* ------------------------------------------------------------------------ */

/*
 * For each of the n (m, j) pairs compute one output of the packed matmul
 * without expanding the matrix: axis 1 sums over the columns of row j,
 * axis 0 over the rows at column j.  x is [M, cols] (axis 1) or [M, rows]
 * (axis 0).  Results: y and a (double [n]).
 */
void tcq_oracle_sample(const uint16_t* x, int64_t M, const uint32_t* codes,
                       int64_t rows, int64_t cols, int bt, int k, int L,
                       int interleave, int axis,
                       const uint16_t* scales, const float* lut,
                       const int64_t* ms, const int64_t* js, int64_t n,
                       double* y, double* a) {
    (void)M;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < n; i++) {
        int64_t m = ms[i], j = js[i];
        double s = 0.0, sa = 0.0;
        if (axis == 1) {
            for (int64_t c = 0; c < cols; c++) {
                uint16_t w = weight_at(codes, rows, cols, bt, k, L, interleave,
                                       scales, lut, j, c, NULL);
                double p = (double)tcq_oracle_bf16_to_float(x[m * cols + c]) *
                           (double)tcq_oracle_bf16_to_float(w);
                s += p;
                sa += fabs(p);
            }
        } else {
            for (int64_t r = 0; r < rows; r++) {
                uint16_t w = weight_at(codes, rows, cols, bt, k, L, interleave,
                                       scales, lut, r, j, NULL);
                double p = (double)tcq_oracle_bf16_to_float(x[m * rows + r]) *
                           (double)tcq_oracle_bf16_to_float(w);
                s += p;
                sa += fabs(p);
            }
        }
        y[i] = s;
        a[i] = sa;
    }
}

/* ------------------------------------------------------------------------ */
/* glue of the synthetic MLP stack (not a step of the method)                */
/* ------------------------------------------------------------------------ */

/*
 * RMSNorm with unit gain: out[m][d] = bf16( x[m][d] / sqrt(mean_d x^2 + eps) ),
 * computed in double.  x, out bf16 [M, D].
 */
void tcq_oracle_rmsnorm(const uint16_t* x, int64_t M, int64_t D, double eps, uint16_t* out) {
    for (int64_t m = 0; m < M; m++) {
        double ss = 0.0;
        for (int64_t d = 0; d < D; d++) {
            double v = (double)tcq_oracle_bf16_to_float(x[m * D + d]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)D + eps);
        for (int64_t d = 0; d < D; d++)
            out[m * D + d] = tcq_oracle_bf16_from_double(
                (double)tcq_oracle_bf16_to_float(x[m * D + d]) * inv);
    }
}

/* SwiGLU gate: out[i] = bf16( silu(g[i]) * u[i] ), silu(v) = v / (1 + e^-v). */
void tcq_oracle_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) {
        double gv = (double)tcq_oracle_bf16_to_float(g[i]);
        double uv = (double)tcq_oracle_bf16_to_float(u[i]);
        out[i] = tcq_oracle_bf16_from_double(gv / (1.0 + exp(-gv)) * uv);
    }
}

/* ------------------------------------------------------------------------ */
/* the unrounded contract                                                    */
/* ------------------------------------------------------------------------ */

/*
 * A second numerical contract: the weight enters the contraction as the f32
 * product of codebook value and row scale, with no bf16 rounding in between
 * (@mlx-bun/inference 1.0.0, kernels/trellis/scatter.ts, the balanced scatter
 * kernels; kernels/trellis/tiled-prefill.ts, the doc comment of the tiled
 * prefill, which names the default matvec's unrounded value as a different
 * contract).
 *   w32[r][c] = f32( lut[win] * f32(scale[r]) )       (float [rows, cols])
 */
void tcq_oracle_expand_f32(const uint32_t* codes, int64_t rows, int64_t cols,
                           int bt, int k, int L, int interleave,
                           const uint16_t* scales, const float* lut, float* w_out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        float s = tcq_oracle_bf16_to_float(scales[r]);
        for (int64_t c = 0; c < cols; c++) {
            int64_t b = c / bt;
            int t = (int)(c % bt);
            const uint32_t* bw = codes + block_base(r, b, rows, cols, bt, k, interleave);
            uint32_t win = tcq_oracle_window(bw, bt, k, L, t);
            w_out[r * cols + c] = (float)((double)lut[win] * (double)s);
        }
    }
}

/* Axis 1 on f32 weights: y[m][r] = sum_c x[m][c] w[r][c] (double), a = sum |.|. */
void tcq_oracle_matmul_axis1_f32w(const uint16_t* x, int64_t M, const float* w,
                                  int64_t rows, int64_t cols, double* y, double* a, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, sa = 0.0;
            for (int64_t c = 0; c < cols; c++) {
                double p = (double)tcq_oracle_bf16_to_float(x[m * cols + c]) * (double)w[r * cols + c];
                s += p;
                sa += fabs(p);
            }
            if (y) y[m * rows + r] = s;
            if (a) a[m * rows + r] = sa;
            if (out) out[m * rows + r] = tcq_oracle_bf16_from_double(s);
        }
    }
}

/* Axis 0 on f32 weights: y[m][c] = sum_r x[m][r] w[r][c] (double), a = sum |.|,
 * and, for splits > 0, the split sums over the same row ranges as the rounded
 * contract's scatter (rp = ceil(rows / splits)). */
void tcq_oracle_matmul_axis0_f32w(const uint16_t* x, int64_t M, const float* w,
                                  int64_t rows, int64_t cols, int64_t splits,
                                  double* y, double* a, uint16_t* out, double* partial) {
    int64_t rp = splits > 0 ? (rows + splits - 1) / splits : rows;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; c++) {
        for (int64_t m = 0; m < M; m++) {
            double s = 0.0, sa = 0.0;
            for (int64_t r = 0; r < rows; r++) {
                double p = (double)tcq_oracle_bf16_to_float(x[m * rows + r]) * (double)w[r * cols + c];
                s += p;
                sa += fabs(p);
            }
            if (y) y[m * cols + c] = s;
            if (a) a[m * cols + c] = sa;
            if (out) out[m * cols + c] = tcq_oracle_bf16_from_double(s);
            if (partial && splits > 0) {
                for (int64_t sp = 0; sp < splits; sp++) {
                    int64_t r0 = sp * rp, r1 = r0 + rp < rows ? r0 + rp : rows;
                    double ps = 0.0;
                    for (int64_t r = r0; r < r1; r++)
                        ps += (double)tcq_oracle_bf16_to_float(x[m * rows + r]) * (double)w[r * cols + c];
                    partial[(m * splits + sp) * cols + c] = ps;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* default split count of the axis-0 scatter                                 */
/* ------------------------------------------------------------------------ */

/*
 * The number of row splits the scatter uses when the caller leaves it open.
 * Up to 4 activation rows: the scatter launch's fixed SCATTER_SPLITS = 128
 * (@mlx-bun/inference 1.0.0, kernels/trellis/scatter.ts).  From 5 rows: the
 * split-K launcher's rule (kernels/trellis/splitk-prefill.ts, the launcher):
 * tilesM = ceil(M/32), tilesN = ceil(cols/32), tilesK = floor(rows/16),
 * ratio = max(1, floor(tilesK / (tilesM * tilesN))),
 * splits = min(32, max(2, 2^ceil(log2(ratio)))).
 * Written with the pages' floating-point formulation.
 */
int64_t tcq_oracle_scatter_default_splits(int64_t rows, int64_t cols, int64_t M) {
    if (M <= 4) return 128;
    double tiles_m = ceil((double)M / 32.0);
    double tiles_n = ceil((double)cols / 32.0);
    double tiles_k = floor((double)rows / 16.0);
    double ratio = floor(tiles_k / (tiles_m * tiles_n));
    if (ratio < 1.0) ratio = 1.0;
    double s = pow(2.0, ceil(log2(ratio)));
    if (s < 2.0) s = 2.0;
    if (s > 32.0) s = 32.0;
    return (int64_t)s;
}
