/*
 * fcm_oracle.c -- plain, slow, fp64 CPU oracle for the fused depthwise/dense k x k -> 1x1
 * pointwise convolution module.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its Python
 * binding) links, loads or calls this file.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA kernels.
 *
 * What it computes, and where the pages define it:
 *  - Depthwise (DW) convolution: one k x k filter per channel, applied over height and
 *    width ("Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs",
 *    section II-B, Figure 2).
 *  - Pointwise (PW) convolution: 1x1 filters spanning all channels (same section).
 *  - A depthwise separable convolution is a DW layer followed by a PW layer (same section).
 *  - Each convolution is followed by its normalization and activation layers; an FCM fuses
 *    up to six layers: two convolutions, each with its norm and activation (section III-A).
 *    With inference-time batch norm folded, norm is a per-channel scale and bias.
 *  - PWDW case (an inverted residual's expansion and depthwise layers): a 1x1 convolution
 *    followed by a depthwise k x k convolution of its output, each with its norm and
 *    activation; the depthwise layer pads its own input, the intermediate, with zeros; the
 *    values of the intermediate under overlapping tiles are recomputed by each tile (the
 *    "_R" of PWDW_R, section II-D, Figure 3(b); sections III-A and IV-B).
 *  - Back-to-back case: a dense 3x3 convolution followed by a 1x1 convolution, each with a
 *    per-channel scale_bias_relu epilogue, NHWC activations ("Fusing two back-to-back
 *    convolutions", CUTLASS discussion #208, the CONV1/CONV2 example).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - zero padding; output size Ho = floor((H + 2p - k) / s) + 1, likewise Wo;
 *  - cross-correlation (no filter flip), output (ho, wo) reads input rows ho*s-p .. ho*s-p+k-1;
 *  - norm+act form is act(scale[c] * acc + bias[c]);
 *  - ReLU = max(v, 0), ReLU6 = min(max(v, 0), 6), none = v;
 *  - the intermediate is kept in fp64 unless a "mirror" rounding of it to the GPU storage
 *    format is requested (used only for diagnosis, never for the parity bar).
 *
 * Layouts (all row-major, innermost last):
 *   x  [N][H][W][C]           input feature maps (NHWC)
 *   wd [C][k][k]              depthwise filters
 *   w1 [K1][k][k][C]          dense conv1 filters (K, R, S, C)
 *   wp [K][Cm]                pointwise filters (Cm = C for DW, K1 for dense)
 *   wq [Cm][C]                PWDW: pointwise filters of the first layer
 *   wd2 [Cm][k][k]            PWDW: depthwise filters of the second layer
 *   m  [N][Ho][Wo][Cm]        intermediate feature maps
 *   y  [N][Ho][Wo][K]         output feature maps
 *
 * Every function returns 0 on success and -1 on an invalid shape.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_RELU = 1, ORACLE_ACT_RELU6 = 2 };
enum { ORACLE_MID_EXACT = 0, ORACLE_MID_F32 = 1, ORACLE_MID_F16 = 2, ORACLE_MID_BF16 = 3 };

/* Activation after the folded norm (section III-A: conv -> norm -> activation). */
static double act_apply(double v, int act) {
    if (act == ORACLE_ACT_RELU) return v > 0.0 ? v : 0.0;
    if (act == ORACLE_ACT_RELU6) {
        if (v < 0.0) return 0.0;
        if (v > 6.0) return 6.0;
        return v;
    }
    return v;
}

/*
 * Round v to the nearest value of a binary floating-point format with `prec` significand
 * bits (implicit bit included), minimum normal exponent `emin` and largest finite value
 * `maxf`, ties to even (IEEE 754 roundTiesToEven).  Values past the largest finite one
 * round to infinity.  f16: prec 11, emin -14.  bf16: prec 8, emin -126.
 */
double oracle_round_format(double v, int prec, int emin, double maxf) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    (void)frexp(v, &e);          /* v = f * 2^e with 0.5 <= |f| < 1: leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < emin) lead = emin; /* subnormal range: fixed quantum 2^(emin - prec + 1) */
    double quantum = ldexp(1.0, lead - (prec - 1));
    double r = nearbyint(v / quantum) * quantum; /* exact scaling; nearbyint ties to even */
    if (fabs(r) > maxf) r = copysign(INFINITY, v);
    return r;
}

static double mid_round(double v, int mid_mode) {
    switch (mid_mode) {
    case ORACLE_MID_F32: return (double)(float)v;
    case ORACLE_MID_F16: return oracle_round_format(v, 11, -14, 65504.0);
    case ORACLE_MID_BF16: return oracle_round_format(v, 8, -126, ldexp(255.0, 120));
    default: return v;
    }
}

static int out_extent(int in, int k, int s, int p) {
    if (k < 1 || s < 1 || p < 0 || in + 2 * p < k) return -1;
    return (in + 2 * p - k) / s + 1;
}

#define IDX4(a, b, c, d, B, C, D) ((((size_t)(a) * (B) + (b)) * (C) + (c)) * (D) + (d))

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Threads the OpenMP runtime will use for the next parallel region (1 without OpenMP). */
int oracle_max_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Depthwise k x k convolution + per-channel scale/bias + activation (section II-B). */
int oracle_dw(int N, int H, int W, int C, int k, int s, int p,
              const double *x, const double *wd, const double *s1, const double *b1, int act1,
              double *m, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int c = 0; c < C; c++) {
                    double t = 0.0;
                    for (int i = 0; i < k; i++) {
                        int hi = ho * s - p + i;
                        if (hi < 0 || hi >= H) continue;
                        for (int j = 0; j < k; j++) {
                            int wi = wo * s - p + j;
                            if (wi < 0 || wi >= W) continue;
                            t += x[IDX4(n, hi, wi, c, H, W, C)] * wd[((size_t)c * k + i) * k + j];
                        }
                    }
                    m[IDX4(n, ho, wo, c, Ho, Wo, C)] = act_apply(s1[c] * t + b1[c], act1);
                }
    return 0;
}

/* Pointwise 1x1 convolution + per-channel scale/bias + activation (section II-B). */
int oracle_pw(int N, int Ho, int Wo, int Cm, int K,
              const double *m, const double *wp, const double *s2, const double *b2, int act2,
              double *y, int nthreads) {
    if (N < 0 || Ho < 1 || Wo < 1 || Cm < 1 || K < 1) return -1;
    set_threads(nthreads);
    long long P = (long long)N * Ho * Wo;
#pragma omp parallel for schedule(static)
    for (long long q = 0; q < P; q++)
        for (int kk = 0; kk < K; kk++) {
            double t = 0.0;
            for (int c = 0; c < Cm; c++) t += m[(size_t)q * Cm + c] * wp[(size_t)kk * Cm + c];
            y[(size_t)q * K + kk] = act_apply(s2[kk] * t + b2[kk], act2);
        }
    return 0;
}

/* Dense k x k convolution C -> K1 + per-channel scale/bias + activation (CONV1 of the
 * back-to-back example). */
int oracle_dense(int N, int H, int W, int C, int K1, int k, int s, int p,
                 const double *x, const double *w1, const double *s1, const double *b1, int act1,
                 double *m, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || K1 < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int j = 0; j < K1; j++) {
                    double t = 0.0;
                    for (int r = 0; r < k; r++) {
                        int hi = ho * s - p + r;
                        if (hi < 0 || hi >= H) continue;
                        for (int u = 0; u < k; u++) {
                            int wi = wo * s - p + u;
                            if (wi < 0 || wi >= W) continue;
                            for (int c = 0; c < C; c++)
                                t += x[IDX4(n, hi, wi, c, H, W, C)] *
                                     w1[IDX4(j, r, u, c, k, k, C)];
                        }
                    }
                    m[IDX4(n, ho, wo, j, Ho, Wo, K1)] = act_apply(s1[j] * t + b1[j], act1);
                }
    return 0;
}

/*
 * The fused module, written as its own single pass: for every output pixel, the first
 * convolution (DW, or dense when `dense` is non-zero) produces that pixel's intermediate
 * vector over all channels, which is then consumed at once by the 1x1 convolution -- the
 * "all channels of the intermediate" requirement of the DWPW case (section II-D).  It does
 * not call oracle_dw/oracle_pw, so comparing the two is a real check.
 * mid_mode: 0 keep the intermediate exact (fp64); 1/2/3 round it to f32/f16/bf16 first.
 */
int oracle_fused(int dense, int N, int H, int W, int C, int Cm, int K, int k, int s, int p,
                 const double *x, const double *w1, const double *s1, const double *b1, int act1,
                 const double *wp, const double *s2, const double *b2, int act2,
                 int mid_mode, double *y, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Cm < 1 || K < 1 || Ho < 1 || Wo < 1) return -1;
    if (!dense && Cm != C) return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double *mid = (double *)malloc(sizeof(double) * (size_t)Cm);
        if (!mid) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for collapse(2) schedule(static)
        for (int n = 0; n < N; n++)
            for (int ho = 0; ho < Ho; ho++) {
                if (!mid) continue;
                for (int wo = 0; wo < Wo; wo++) {
                    for (int j = 0; j < Cm; j++) {
                        double t = 0.0;
                        for (int r = 0; r < k; r++) {
                            int hi = ho * s - p + r;
                            if (hi < 0 || hi >= H) continue;
                            for (int u = 0; u < k; u++) {
                                int wi = wo * s - p + u;
                                if (wi < 0 || wi >= W) continue;
                                if (dense) {
                                    for (int c = 0; c < C; c++)
                                        t += x[IDX4(n, hi, wi, c, H, W, C)] *
                                             w1[IDX4(j, r, u, c, k, k, C)];
                                } else {
                                    t += x[IDX4(n, hi, wi, j, H, W, C)] *
                                         w1[((size_t)j * k + r) * k + u];
                                }
                            }
                        }
                        mid[j] = mid_round(act_apply(s1[j] * t + b1[j], act1), mid_mode);
                    }
                    for (int kk = 0; kk < K; kk++) {
                        double t = 0.0;
                        for (int j = 0; j < Cm; j++) t += mid[j] * wp[(size_t)kk * Cm + j];
                        y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = act_apply(s2[kk] * t + b2[kk], act2);
                    }
                }
            }
        free(mid);
    }
    return failed ? -1 : 0;
}

/*
 * The PWDW module as its own single pass: for every output pixel and channel j, the value of
 * the intermediate under each depthwise tap is the 1x1 convolution of the input pixel there,
 * recomputed on the spot, followed by its norm and activation (and the optional mirror
 * rounding); taps that fall in the padding read zero, because the padding belongs to the
 * depthwise layer's input.  It does not call oracle_pw/oracle_dw.
 * x [N][H][W][C], wq [Cm][C], wd2 [Cm][k][k] -> y [N][Ho][Wo][Cm].
 */
int oracle_pwdw(int N, int H, int W, int C, int Cm, int k, int s, int p,
                const double *x, const double *wq, const double *s1, const double *b1, int act1,
                const double *wd2, const double *s2, const double *b2, int act2,
                int mid_mode, double *y, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Cm < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int j = 0; j < Cm; j++) {
                    double t = 0.0;
                    for (int i = 0; i < k; i++) {
                        int hi = ho * s - p + i;
                        if (hi < 0 || hi >= H) continue;
                        for (int u = 0; u < k; u++) {
                            int wi = wo * s - p + u;
                            if (wi < 0 || wi >= W) continue;
                            double q = 0.0;
                            for (int c = 0; c < C; c++)
                                q += x[IDX4(n, hi, wi, c, H, W, C)] * wq[(size_t)j * C + c];
                            double mval = mid_round(act_apply(s1[j] * q + b1[j], act1), mid_mode);
                            t += mval * wd2[((size_t)j * k + i) * k + u];
                        }
                    }
                    y[IDX4(n, ho, wo, j, Ho, Wo, Cm)] = act_apply(s2[j] * t + b2[j], act2);
                }
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * INT8 module (section III-B: INT8 feature maps and weights, four-way int8 products with
 * 32-bit accumulation, every buffer -- the commBuffer included -- holding int8 values packed
 * four to a word; weights packed offline).  The pages give no quantization scheme, so the
 * plainest one is read (and listed in the design notes):
 *  - x, the filters, the intermediate m and the output y are int8; a convolution's
 *    accumulator is the exact integer sum of int8 x int8 products;
 *  - the folded norm is a per-channel fp32 scale and bias, applied to the accumulator as one
 *    fp32 fused multiply-add, v = fma(s, (float)acc, b) (|acc| < 2^24 for every supported
 *    shape, so the conversion is exact); this is the precision in which the GPU takes the
 *    rounding decision, so the oracle takes it in the same one;
 *  - then the activation, rounding to the nearest integer (ties to even) and saturation to
 *    [-128, 127]: q = clamp(rint(act(v)), -128, 127).
 * The accumulators are int64 here, so nothing can overflow.
 * Layouts as above: x [N][H][W][C], wd [C][k][k], wp [K][C], m [N][Ho][Wo][C],
 * y [N][Ho][Wo][K]; s and b are float32.
 * ------------------------------------------------------------------------------------------ */

/* Requantization of one accumulator to int8. */
static int8_t requant_i8(int64_t acc, float s, float b, int act) {
    float v = fmaf(s, (float)acc, b);
    double a = act_apply((double)v, act);
    double r = nearbyint(a); /* default rounding mode: to nearest, ties to even */
    if (r < -128.0) r = -128.0;
    if (r > 127.0) r = 127.0;
    return (int8_t)r;
}

/* Requantization of one value, exposed for the tests' closed-form checks. */
int oracle_requant_i8(long long acc, float s, float b, int act) {
    return (int)requant_i8((int64_t)acc, s, b, act);
}

/* INT8 depthwise k x k convolution + requantization (section II-B, section III-B INT8). */
int oracle_dw_i8(int N, int H, int W, int C, int k, int s, int p,
                 const int8_t *x, const int8_t *wd, const float *s1, const float *b1, int act1,
                 int8_t *m, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int c = 0; c < C; c++) {
                    int64_t t = 0;
                    for (int i = 0; i < k; i++) {
                        int hi = ho * s - p + i;
                        if (hi < 0 || hi >= H) continue;
                        for (int j = 0; j < k; j++) {
                            int wi = wo * s - p + j;
                            if (wi < 0 || wi >= W) continue;
                            t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *
                                 (int64_t)wd[((size_t)c * k + i) * k + j];
                        }
                    }
                    m[IDX4(n, ho, wo, c, Ho, Wo, C)] = requant_i8(t, s1[c], b1[c], act1);
                }
    return 0;
}

/* INT8 pointwise 1x1 convolution + requantization. */
int oracle_pw_i8(int N, int Ho, int Wo, int Cm, int K,
                 const int8_t *m, const int8_t *wp, const float *s2, const float *b2, int act2,
                 int8_t *y, int nthreads) {
    if (N < 0 || Ho < 1 || Wo < 1 || Cm < 1 || K < 1) return -1;
    set_threads(nthreads);
    long long P = (long long)N * Ho * Wo;
#pragma omp parallel for schedule(static)
    for (long long q = 0; q < P; q++)
        for (int kk = 0; kk < K; kk++) {
            int64_t t = 0;
            for (int c = 0; c < Cm; c++)
                t += (int64_t)m[(size_t)q * Cm + c] * (int64_t)wp[(size_t)kk * Cm + c];
            y[(size_t)q * K + kk] = requant_i8(t, s2[kk], b2[kk], act2);
        }
    return 0;
}

/* The INT8 DW -> PW module as its own single pass (one output pixel at a time: its int8
 * intermediate vector over all channels, then the 1x1 convolution of it).  It does not call
 * oracle_dw_i8/oracle_pw_i8. */
int oracle_fused_i8(int N, int H, int W, int C, int K, int k, int s, int p,
                    const int8_t *x, const int8_t *wd, const float *s1, const float *b1, int act1,
                    const int8_t *wp, const float *s2, const float *b2, int act2,
                    int8_t *y, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || K < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        int8_t *mid = (int8_t *)malloc((size_t)C);
        if (!mid) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for collapse(2) schedule(static)
        for (int n = 0; n < N; n++)
            for (int ho = 0; ho < Ho; ho++) {
                if (!mid) continue;
                for (int wo = 0; wo < Wo; wo++) {
                    for (int c = 0; c < C; c++) {
                        int64_t t = 0;
                        for (int i = 0; i < k; i++) {
                            int hi = ho * s - p + i;
                            if (hi < 0 || hi >= H) continue;
                            for (int j = 0; j < k; j++) {
                                int wi = wo * s - p + j;
                                if (wi < 0 || wi >= W) continue;
                                t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *
                                     (int64_t)wd[((size_t)c * k + i) * k + j];
                            }
                        }
                        mid[c] = requant_i8(t, s1[c], b1[c], act1);
                    }
                    for (int kk = 0; kk < K; kk++) {
                        int64_t t = 0;
                        for (int c = 0; c < C; c++)
                            t += (int64_t)mid[c] * (int64_t)wp[(size_t)kk * C + c];
                        y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = requant_i8(t, s2[kk], b2[kk], act2);
                    }
                }
            }
        free(mid);
    }
    return failed ? -1 : 0;
}

/* INT8 dense k x k convolution C -> Cm + requantization (the back-to-back CONV1; with k = 1
 * the first layer of the PWPW module).  w1 [Cm][k][k][C]. */
int oracle_dense_i8(int N, int H, int W, int C, int Cm, int k, int s, int p,
                    const int8_t *x, const int8_t *w1, const float *s1, const float *b1, int act1,
                    int8_t *m, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Cm < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int j = 0; j < Cm; j++) {
                    int64_t t = 0;
                    for (int r = 0; r < k; r++) {
                        int hi = ho * s - p + r;
                        if (hi < 0 || hi >= H) continue;
                        for (int u = 0; u < k; u++) {
                            int wi = wo * s - p + u;
                            if (wi < 0 || wi >= W) continue;
                            for (int c = 0; c < C; c++)
                                t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *
                                     (int64_t)w1[IDX4(j, r, u, c, k, k, C)];
                        }
                    }
                    m[IDX4(n, ho, wo, j, Ho, Wo, Cm)] = requant_i8(t, s1[j], b1[j], act1);
                }
    return 0;
}

/* The INT8 dense k x k -> 1x1 module (PWPW when k = 1) as its own single pass: one output
 * pixel at a time, its int8 intermediate vector over all Cm channels, then the 1x1
 * convolution of it.  It does not call oracle_dense_i8/oracle_pw_i8. */
int oracle_fused_dense_i8(int N, int H, int W, int C, int Cm, int K, int k, int s, int p,
                          const int8_t *x, const int8_t *w1, const float *s1, const float *b1,
                          int act1, const int8_t *wp, const float *s2, const float *b2, int act2,
                          int8_t *y, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Cm < 1 || K < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        int8_t *mid = (int8_t *)malloc((size_t)Cm);
        if (!mid) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for collapse(2) schedule(static)
        for (int n = 0; n < N; n++)
            for (int ho = 0; ho < Ho; ho++) {
                if (!mid) continue;
                for (int wo = 0; wo < Wo; wo++) {
                    for (int j = 0; j < Cm; j++) {
                        int64_t t = 0;
                        for (int r = 0; r < k; r++) {
                            int hi = ho * s - p + r;
                            if (hi < 0 || hi >= H) continue;
                            for (int u = 0; u < k; u++) {
                                int wi = wo * s - p + u;
                                if (wi < 0 || wi >= W) continue;
                                for (int c = 0; c < C; c++)
                                    t += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *
                                         (int64_t)w1[IDX4(j, r, u, c, k, k, C)];
                            }
                        }
                        mid[j] = requant_i8(t, s1[j], b1[j], act1);
                    }
                    for (int kk = 0; kk < K; kk++) {
                        int64_t t = 0;
                        for (int j = 0; j < Cm; j++)
                            t += (int64_t)mid[j] * (int64_t)wp[(size_t)kk * Cm + j];
                        y[IDX4(n, ho, wo, kk, Ho, Wo, K)] = requant_i8(t, s2[kk], b2[kk], act2);
                    }
                }
            }
        free(mid);
    }
    return failed ? -1 : 0;
}

/* The INT8 PWDW module as its own single pass (section II-D's PWDW with section III-B's INT8
 * buffers): for every output pixel and channel j, the int8 intermediate under each depthwise
 * tap is the 1x1 convolution of the input pixel there, requantized on the spot; taps that
 * fall in the padding read int8 zero, because the padding belongs to the depthwise layer's
 * input.  It does not call oracle_pw_i8/oracle_dw_i8.
 * x [N][H][W][C], wq [Cm][C], wd2 [Cm][k][k] int8; s1/b1, s2/b2 [Cm] -> y [N][Ho][Wo][Cm]. */
int oracle_pwdw_i8(int N, int H, int W, int C, int Cm, int k, int s, int p,
                   const int8_t *x, const int8_t *wq, const float *s1, const float *b1, int act1,
                   const int8_t *wd2, const float *s2, const float *b2, int act2,
                   int8_t *y, int nthreads) {
    int Ho = out_extent(H, k, s, p), Wo = out_extent(W, k, s, p);
    if (N < 0 || C < 1 || Cm < 1 || Ho < 1 || Wo < 1) return -1;
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; n++)
        for (int ho = 0; ho < Ho; ho++)
            for (int wo = 0; wo < Wo; wo++)
                for (int j = 0; j < Cm; j++) {
                    int64_t t = 0;
                    for (int i = 0; i < k; i++) {
                        int hi = ho * s - p + i;
                        if (hi < 0 || hi >= H) continue;
                        for (int u = 0; u < k; u++) {
                            int wi = wo * s - p + u;
                            if (wi < 0 || wi >= W) continue;
                            int64_t q = 0;
                            for (int c = 0; c < C; c++)
                                q += (int64_t)x[IDX4(n, hi, wi, c, H, W, C)] *
                                     (int64_t)wq[(size_t)j * C + c];
                            int8_t mval = requant_i8(q, s1[j], b1[j], act1);
                            t += (int64_t)mval * (int64_t)wd2[((size_t)j * k + i) * k + u];
                        }
                    }
                    y[IDX4(n, ho, wo, j, Ho, Wo, Cm)] = requant_i8(t, s2[j], b2[j], act2);
                }
    return 0;
}
