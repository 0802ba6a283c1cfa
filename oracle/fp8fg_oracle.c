/*
 * fp8fg_oracle.c -- plain, slow CPU oracle for fine-grained FP8 quantization
 * and the block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check of the
 * entry module and the benchmark's CPU-baseline leg may load this library.
 * The product path (the CUDA library under fp8_fine_grained_act_gb300/) never
 * calls it, includes none of its code and shares no header with it.
 *
 * What it computes, and where it comes from:
 *   - E4M3 decode/encode: the 8-bit format with a 4-bit exponent and a 3-bit
 *     mantissa ("FP8 Mixed-Precision Training: Hardware Acceleration Beyond
 *     NVIDIA's Paradigm", section 1.1); the E4M3 variant with maximum 448
 *     (OCP 8-bit floating point specification, E4M3: bias 7, no infinities,
 *     S.1111.111 is NaN).  Encoding rounds to nearest, ties to even, and
 *     saturates to +-448 ("scaling the maximum absolute value of the input to
 *     the maximum representable value of FP8", DeepSeek-V3 FP8 post on
 *     innerforce.co.kr, fine-grained quantization paragraph).
 *   - Group scales: one FP32 scale per group, computed online from the
 *     current group's maximum absolute value ("Unified E4M3 format in
 *     DeepSeek-V3", codingmall.com, section "Dynamic Scaling and Online
 *     Quantization"), s = amax / 448 in IEEE single precision.
 *   - Group geometry: 1x128 tiles per token per 128 channels for activations,
 *     128x128 blocks for weights (innerforce.co.kr post, Figure 7 (a);
 *     "DeepSeek FP8 Training", arcalunar.github.io, tile-wise 1 x N_c and
 *     block-wise N_c x N_c grouping, N_c = 128).  The 128x1 token-axis mode
 *     groups 128 consecutive tokens of one channel for the weight-gradient
 *     GEMM, whose reduction runs over tokens ("DeepSeek FP8 Training",
 *     backward pass, Wgrad step 1).
 *   - GEMM: o[i,j] = sum_k a~[i,k] * b~[j,k] with a~ = dec(q_a) * s_a,
 *     b~ = dec(q_b) * s_b, summed in double, plus the magnitude sum
 *     m[i,j] = sum_k |a~[i,k] * b~[j,k]| that the GPU tolerance is stated in.
 *     This is the plain definition of what the per-128-chunk scaled and
 *     promoted FP8 GEMM computes ("DeepSeek FP8 Training", forward steps 3-4;
 *     "Unified E4M3 format in DeepSeek-V3", section "Enhanced Numerical
 *     Stability").
 *
 * Readings taken where the pages are silent: the element code is
 * enc(fl32(x / s)) with an IEEE single division (the pages give only
 * "scale = amax / 448" and the quantize step; a multiply by a reciprocal
 * and x * fl(448 / amax) differ from it in the last bit on rare inputs);
 * a group whose scale is 0 (all zeros, or amax / 448 underflowing in FP32)
 * stores s = 0 and codes that keep only the sign of x, so it dequantizes to
 * zero; NaN input encodes to 0x7F with its sign bit (parity unpinned:
 * inputs are finite by precondition).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp -ffp-contract=off
 *        -fno-fast-math (no FMA contraction, IEEE single division).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FO_GROUP 128

/* ---------------------------------------------------------------- E4M3 --- */

/* Value of an E4M3 code: sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0.  Exponent field 0 is subnormal: (m/8) * 2^-6.  0x7F and 0xFF
 * are NaN.  Every finite value is returned exactly. */
double fo_e4m3_decode(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-half-to-even of a non-negative double.  Callers pass |v| / step with
 * step a power of two, so the argument is exact and at most 2^4. */
static double fo_round_half_even(double n)
{
    double f = floor(n);
    double d = n - f;
    if (d > 0.5)
        return f + 1.0;
    if (d < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* E4M3 code of an FP32 value: round to the nearest point of the E4M3 grid,
 * ties to an even mantissa; magnitudes above 448 (including infinity) become
 * 448; zero and results that round to zero keep the sign of v. */
uint8_t fo_e4m3_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a > 448.0)
        return (uint8_t)(sign | 0x7E);
    /* Grid step: 2^-9 below the smallest normal 2^-6, else 2^(e-3) in the
     * binade [2^e, 2^(e+1)). */
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);
    } else {
        int e2;
        frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) -> binade e2-1 */
        step = ldexp(1.0, (e2 - 1) - 3);
    }
    double r = fo_round_half_even(a / step) * step;   /* a / step is exact */
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    int E, M;
    if (r < ldexp(1.0, -6)) {
        E = 0;
        M = (int)(r / ldexp(1.0, -9));
    } else {
        int e2;
        double f = frexp(r, &e2);   /* r = f * 2^e2 */
        E = (e2 - 1) + 7;
        M = (int)(f * 16.0 - 8.0);  /* f*2 = 1 + M/8 */
    }
    return (uint8_t)(sign | (E << 3) | M);
}

void fo_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fo_e4m3_encode(v[i]);
}

void fo_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fo_e4m3_decode(c[i]);
}

/* ------------------------------------------------------- group quantize --- */

static float fo_bf16_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Quantize one group of n values given as FP32 (read through a stride):
 * amax -> s = fl32(amax / 448) -> q = enc(fl32(x / s)).  A zero scale gives
 * codes that keep only the sign of x. */
static float fo_quant_group(const float *x, int64_t n, int64_t stride_x,
                            uint8_t *q, int64_t stride_q)
{
    float amax = 0.0f;
    for (int64_t t = 0; t < n; ++t) {
        float ax = fabsf(x[t * stride_x]);
        if (ax > amax)
            amax = ax;
    }
    volatile float s = amax / 448.0f;      /* IEEE single division */
    for (int64_t t = 0; t < n; ++t) {
        float xv = x[t * stride_x];
        if (s == 0.0f) {
            uint32_t bits;
            memcpy(&bits, &xv, sizeof bits);
            q[t * stride_q] = (uint8_t)((bits >> 31) << 7);
        } else {
            volatile float qv = xv / s;    /* IEEE single division */
            q[t * stride_q] = fo_e4m3_encode(qv);
        }
    }
    return s;
}

/* Activations / gradients, BF16 input x[rows, cols] (row-major, bits given as
 * uint16).
 *   axis 0 (1x128, per token per 128 channels): cols % 128 == 0;
 *     q[rows, cols], s[cols/128, rows] with s[c*rows + i] for group
 *     x[i, 128c .. 128c+127].
 *   axis 1 (128x1, 128 consecutive tokens of one channel): rows % 128 == 0;
 *     q is written transposed, q[cols, rows]; s[rows/128, cols] with
 *     s[t*cols + j] for group x[128t .. 128t+127, j].
 * Returns 0, or -1 for a shape that does not tile into whole groups. */
int fo_quant_act(const uint16_t *x, int64_t rows, int64_t cols, int axis,
                 uint8_t *q, float *s)
{
    float buf[FO_GROUP];
    uint8_t qb[FO_GROUP];
    if (axis == 0) {
        if (cols % FO_GROUP)
            return -1;
        int64_t ng = cols / FO_GROUP;
        for (int64_t i = 0; i < rows; ++i)
            for (int64_t c = 0; c < ng; ++c) {
                for (int t = 0; t < FO_GROUP; ++t)
                    buf[t] = fo_bf16_to_float(x[i * cols + c * FO_GROUP + t]);
                s[c * rows + i] = fo_quant_group(buf, FO_GROUP, 1, qb, 1);
                for (int t = 0; t < FO_GROUP; ++t)
                    q[i * cols + c * FO_GROUP + t] = qb[t];
            }
        return 0;
    }
    if (axis == 1) {
        if (rows % FO_GROUP)
            return -1;
        int64_t ng = rows / FO_GROUP;
        for (int64_t tb = 0; tb < ng; ++tb)
            for (int64_t j = 0; j < cols; ++j) {
                for (int t = 0; t < FO_GROUP; ++t)
                    buf[t] = fo_bf16_to_float(x[(tb * FO_GROUP + t) * cols + j]);
                s[tb * cols + j] = fo_quant_group(buf, FO_GROUP, 1, qb, 1);
                for (int t = 0; t < FO_GROUP; ++t)
                    q[j * rows + tb * FO_GROUP + t] = qb[t];
            }
        return 0;
    }
    return -1;
}

/* FP32 master weight w[rows, cols] in 128x128 blocks (rows % 128 == 0,
 * cols % 128 == 0).  q[rows, cols]; q_t (may be NULL) receives the same codes
 * transposed, q_t[cols, rows]; s[rows/128, cols/128] row-major. */
int fo_quant_w(const float *w, int64_t rows, int64_t cols,
               uint8_t *q, uint8_t *q_t, float *s)
{
    if (rows % FO_GROUP || cols % FO_GROUP)
        return -1;
    int64_t nbr = rows / FO_GROUP, nbc = cols / FO_GROUP;
    static float blk[FO_GROUP * FO_GROUP];
    static uint8_t qb[FO_GROUP * FO_GROUP];
    for (int64_t r = 0; r < nbr; ++r)
        for (int64_t c = 0; c < nbc; ++c) {
            for (int i = 0; i < FO_GROUP; ++i)
                for (int j = 0; j < FO_GROUP; ++j)
                    blk[i * FO_GROUP + j] =
                        w[(r * FO_GROUP + i) * cols + c * FO_GROUP + j];
            s[r * nbc + c] = fo_quant_group(blk, FO_GROUP * FO_GROUP, 1, qb, 1);
            for (int i = 0; i < FO_GROUP; ++i)
                for (int j = 0; j < FO_GROUP; ++j) {
                    int64_t gi = r * FO_GROUP + i, gj = c * FO_GROUP + j;
                    q[gi * cols + gj] = qb[i * FO_GROUP + j];
                    if (q_t)
                        q_t[gj * rows + gi] = qb[i * FO_GROUP + j];
                }
        }
    return 0;
}

/* ------------------------------------------------------------------ GEMM --- */

/* B-operand scale of element (j, k):
 *   bscale 0 (128x128 blocks): sb[(j/128)*stride_n + (k/128)*stride_k];
 *   bscale 1 (per row, per 128-wide K chunk): sb[(k/128)*N + j]. */
static double fo_sb(const float *sb, int bscale, int64_t stride_n,
                    int64_t stride_k, int64_t N, int64_t j, int64_t k)
{
    if (bscale == 0)
        return (double)sb[(j / FO_GROUP) * stride_n + (k / FO_GROUP) * stride_k];
    return (double)sb[(k / FO_GROUP) * N + j];
}

/* D = A . B^T for the listed entries (ei[e], ej[e]).
 * A: q_a[M, K] codes, s_a[K/128, M];  B: q_b[N, K] codes, scales per bscale.
 * o[e] = sum_k a~[i,k] b~[j,k] and m[e] = sum_k |a~[i,k] b~[j,k]|, in double,
 * k ascending. */
void fo_gemm_entries(const uint8_t *qa, const float *sa, int64_t M,
                     const uint8_t *qb, const float *sb, int bscale,
                     int64_t sb_stride_n, int64_t sb_stride_k, int64_t N,
                     int64_t K, int64_t n_entries, const int64_t *ei,
                     const int64_t *ej, double *o, double *m)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < n_entries; ++e) {
        int64_t i = ei[e], j = ej[e];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = fo_e4m3_decode(qa[i * K + k]) *
                       (double)sa[(k / FO_GROUP) * M + i];
            double b = fo_e4m3_decode(qb[j * K + k]) *
                       fo_sb(sb, bscale, sb_stride_n, sb_stride_k, N, j, k);
            double p = a * b;
            acc += p;
            mag += fabs(p);
        }
        o[e] = acc;
        m[e] = mag;
    }
}

/* The whole output o[M, N], m[M, N] (row-major).  The operands are first
 * dequantized into double matrices (a~ and b~ are exact in double), then the
 * dot products are taken row by row. */
void fo_gemm_full(const uint8_t *qa, const float *sa, int64_t M,
                  const uint8_t *qb, const float *sb, int bscale,
                  int64_t sb_stride_n, int64_t sb_stride_k, int64_t N,
                  int64_t K, double *a_deq, double *b_deq, double *o, double *m)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k)
            a_deq[i * K + k] = fo_e4m3_decode(qa[i * K + k]) *
                               (double)sa[(k / FO_GROUP) * M + i];
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            b_deq[j * K + k] = fo_e4m3_decode(qb[j * K + k]) *
                               fo_sb(sb, bscale, sb_stride_n, sb_stride_k, N, j, k);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            const double *ar = a_deq + i * K, *br = b_deq + j * K;
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ar[k] * br[k];
                acc += p;
                mag += fabs(p);
            }
            o[i * N + j] = acc;
            m[i * N + j] = mag;
        }
}

int fo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void fo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
