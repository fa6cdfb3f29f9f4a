/*
 * om_oracle.c -- plain, slow, obviously correct CPU oracle for the fp32
 * matrix product and the NCHW 2-D convolution.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code, header, table or constant
 * with the CUDA library; it is compiled on its own with
 *     -O2 -ffp-contract=off -fno-fast-math
 * so that no multiply and add are ever contracted into a fused operation
 * and every float operation is one IEEE binary32 operation with
 * round-to-nearest-even (the host's default rounding and subnormal modes;
 * oracle_selfcheck() verifies both at run time).
 *
 * Sources (OneModel documentation pages):
 *  - "Exact mode", section "Matrix product (C = A * B, row-major ...)":
 *    per output acc = +0; for p = 0..k-1 in increasing order,
 *    prod = round(A[i][p] * B[p][j]); acc = round(acc + prod); a NaN result
 *    is stored as the bits 0x7FC00000; k = 0 gives +0.
 *  - "Exact mode", section "Rules every exact kernel follows" (rules 1-4:
 *    RNE binary32, no fused multiply-add, no flush-to-zero, start from +0,
 *    canonical NaN).
 *  - "Matrix product and convolution kernels", section "Fast mode": the same
 *    order with one fused multiply-add per term.
 *  - "Exact mode", section "Convolution (2-D, NCHW, weights [Cout, Cin/G,
 *    KH, KW])": the tap loop (channel, kernel row, kernel column), the input
 *    coordinates, the +0 value outside the plane (padding taps are real
 *    products), and the output-size formula.
 *
 * Reading taken where the pages leave it open: fast mode also stores every
 * NaN as 0x7FC00000 (the pages let fast mode keep the hardware payload;
 * canonicalising both modes makes them bit-comparable).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

#define ORACLE_MODE_EXACT 0
#define ORACLE_MODE_FAST 1

int oracle_abi_version(void) { return 1; }

/* Store rule of both modes: a NaN accumulator becomes the quiet NaN 0x7FC00000. */
static float canonical(float acc) {
    if (isnan(acc)) {
        const uint32_t q = 0x7FC00000u;
        float out;
        memcpy(&out, &q, sizeof out);
        return out;
    }
    return acc;
}

/* One term of an output's sum, in the mode's arithmetic. */
static float add_term(float acc, float a, float b, int mode) {
    if (mode == ORACLE_MODE_FAST) {
        return fmaf(a, b, acc);        /* one rounding: round(a*b + acc) */
    }
    float prod = a * b;                /* rounded to binary32 */
    return acc + prod;                 /* rounded to binary32 */
}

/*
 * Returns 0 when the host computes binary32 with subnormals kept and no
 * excess precision; a positive code names the first check that failed.
 */
int oracle_selfcheck(void) {
    volatile float tiny = 1e-40f, one = 1.0f;
    if (tiny * one == 0.0f) return 1;                       /* flush-to-zero */
    volatile float big = 16777216.0f;                       /* 2^24 */
    if (big + one != big) return 2;                         /* excess precision */
    volatile float a = 1.0f + 1.0f / 4096.0f, m1 = -1.0f;
    float e = add_term(add_term(0.0f, m1, one, 0), a, a, 0);
    float f = add_term(add_term(0.0f, m1, one, 1), a, a, 1);
    if (e != 1.0f / 2048.0f) return 3;                      /* contraction in exact mode */
    if (f != 1.0f / 2048.0f + 1.0f / 16777216.0f) return 4; /* fmaf not fused */
    return 0;
}

/*
 * C = A * B, row-major, A is m x k (row stride lda), B is k x n (ldb),
 * C is m x n (ldc). Only C[i][j] with i < m, j < n is written.
 * threads > 1 spreads whole rows over OpenMP threads; every output is
 * computed by one thread over all of k, so the count cannot change a bit.
 */
void oracle_gemm_f32(int64_t m, int64_t n, int64_t k,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float *C, int64_t ldc, int mode, int threads) {
    (void)threads;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            float acc = +0.0f;
            for (int64_t p = 0; p < k; ++p) {
                acc = add_term(acc, A[i * lda + p], B[p * ldb + j], mode);
            }
            C[i * ldc + j] = canonical(acc);
        }
    }
}

/*
 * Output size per axis: floor((size + pad_before + pad_after
 * - dilation*(K-1) - 1) / stride) + 1, taken as 0 when that is not positive.
 */
int64_t oracle_conv_out_dim(int64_t size, int64_t ksize, int64_t stride,
                            int64_t pad_before, int64_t pad_after, int64_t dil) {
    int64_t num = size + pad_before + pad_after - dil * (ksize - 1) - 1;
    if (stride < 1 || num < 0) return 0;
    return num / stride + 1;
}

/*
 * 2-D convolution, NCHW. x is [N][Cin][H][W], w is [Cout][Cin/G][KH][KW],
 * y is [N][Cout][OutH][OutW], all contiguous. Output (n, oc, oy, ox) of
 * group g = oc / (Cout/G) sums, for c, then ky, then kx in increasing order,
 * w[oc][c][ky][kx] * v with iy = oy*sH - pT + ky*dH, ix = ox*sW - pL + kx*dW
 * and v = x[n][g*Cin/G + c][iy][ix] inside the plane, +0 outside.
 */
void oracle_conv2d_f32(int64_t N, int64_t Cin, int64_t H, int64_t W,
                       int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pT, int64_t pL,
                       int64_t pB, int64_t pR, int64_t dH, int64_t dW,
                       const float *x, const float *w, float *y,
                       int mode, int threads) {
    (void)threads;
    const int64_t OH = oracle_conv_out_dim(H, KH, sH, pT, pB, dH);
    const int64_t OW = oracle_conv_out_dim(W, KW, sW, pL, pR, dW);
    const int64_t cin_g = Cin / G, cout_g = Cout / G;
#pragma omp parallel for collapse(2) schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t oc = 0; oc < Cout; ++oc) {
            const int64_t g = oc / cout_g;
            for (int64_t oy = 0; oy < OH; ++oy) {
                for (int64_t ox = 0; ox < OW; ++ox) {
                    float acc = +0.0f;
                    for (int64_t c = 0; c < cin_g; ++c) {
                        for (int64_t ky = 0; ky < KH; ++ky) {
                            for (int64_t kx = 0; kx < KW; ++kx) {
                                const int64_t iy = oy * sH - pT + ky * dH;
                                const int64_t ix = ox * sW - pL + kx * dW;
                                float v = +0.0f;
                                if (iy >= 0 && iy < H && ix >= 0 && ix < W) {
                                    v = x[((n * Cin + g * cin_g + c) * H + iy) * W + ix];
                                }
                                const float wt = w[((oc * cin_g + c) * KH + ky) * KW + kx];
                                acc = add_term(acc, wt, v, mode);
                            }
                        }
                    }
                    y[((n * Cout + oc) * OH + oy) * OW + ox] = canonical(acc);
                }
            }
        }
    }
}

/*
 * Double-precision companions used only for error bounds: for each output,
 * ref = sum_p a_p*b_p and mag = sum_p |a_p*b_p| in increasing p, in binary64.
 */
void oracle_gemm_f64(int64_t m, int64_t n, int64_t k,
                     const float *A, int64_t lda, const float *B, int64_t ldb,
                     double *ref, double *mag, int64_t ldc, int threads) {
    (void)threads;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double s = 0.0, t = 0.0;
            for (int64_t p = 0; p < k; ++p) {
                const double prod = (double)A[i * lda + p] * (double)B[p * ldb + j];
                s = s + prod;
                t = t + fabs(prod);
            }
            ref[i * ldc + j] = s;
            mag[i * ldc + j] = t;
        }
    }
}

void oracle_conv2d_f64(int64_t N, int64_t Cin, int64_t H, int64_t W,
                       int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                       int64_t sH, int64_t sW, int64_t pT, int64_t pL,
                       int64_t pB, int64_t pR, int64_t dH, int64_t dW,
                       const float *x, const float *w, double *ref, double *mag,
                       int threads) {
    (void)threads;
    const int64_t OH = oracle_conv_out_dim(H, KH, sH, pT, pB, dH);
    const int64_t OW = oracle_conv_out_dim(W, KW, sW, pL, pR, dW);
    const int64_t cin_g = Cin / G, cout_g = Cout / G;
#pragma omp parallel for collapse(2) schedule(static) num_threads(threads > 0 ? threads : 1)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t oc = 0; oc < Cout; ++oc) {
            const int64_t g = oc / cout_g;
            for (int64_t oy = 0; oy < OH; ++oy) {
                for (int64_t ox = 0; ox < OW; ++ox) {
                    double s = 0.0, t = 0.0;
                    for (int64_t c = 0; c < cin_g; ++c) {
                        for (int64_t ky = 0; ky < KH; ++ky) {
                            for (int64_t kx = 0; kx < KW; ++kx) {
                                const int64_t iy = oy * sH - pT + ky * dH;
                                const int64_t ix = ox * sW - pL + kx * dW;
                                double v = 0.0;
                                if (iy >= 0 && iy < H && ix >= 0 && ix < W) {
                                    v = x[((n * Cin + g * cin_g + c) * H + iy) * W + ix];
                                }
                                const double prod = (double)w[((oc * cin_g + c) * KH + ky) * KW + kx] * v;
                                s = s + prod;
                                t = t + fabs(prod);
                            }
                        }
                    }
                    const int64_t o = ((n * Cout + oc) * OH + oy) * OW + ox;
                    ref[o] = s;
                    mag[o] = t;
                }
            }
        }
    }
}

/*
 * Output epilogue ("Convolution (fast mode)", section "Tiles and chunks": the
 * epilogue, bias then activation, applied to each finished tile, rows counted
 * from the group's first output channel; section "Single-column products":
 * the bias, activation and residual epilogue). The pages do not fix where the
 * residual goes relative to the activation; the reading taken here is bias,
 * then residual, then activation, each one binary32 operation:
 *   v = y; v = v + bias[ch]; v = v + res; v = relu(v); store canonical(v)
 * with relu(v) = v for v > 0 or NaN, +0 otherwise (so relu(-0) = +0).
 * y holds `count` outputs; output o belongs to channel (o / plane) % channels
 * (plane = OH*OW, channels = Cout for a convolution; plane = 1, channels = n
 * for a row-major m x n product, where the bias is per column). bias and res
 * may be NULL; res has y's layout. activation: 0 none, 1 ReLU.
 */
void oracle_epilogue_f32(int64_t count, int64_t plane, int64_t channels, float *y,
                         const float *bias, const float *res, int activation) {
    for (int64_t o = 0; o < count; ++o) {
        float v = y[o];
        if (bias) v = v + bias[(o / plane) % channels];
        if (res) v = v + res[o];
        if (activation == 1 && !(v > 0.0f) && !isnan(v)) v = +0.0f;
        y[o] = canonical(v);
    }
}
