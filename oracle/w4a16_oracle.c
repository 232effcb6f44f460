/*
 * w4a16_oracle.c -- plain, slow, obviously correct CPU oracle for the W4A16
 * weight-only linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library; both are written independently from the format description.
 *
 * What it computes, and where the pages say so:
 *
 *  - Weight-only quantisation keeps activations and accumulators in 16/32-bit
 *    and stores only the weights in low precision, as small integers per group
 *    plus a scale and a zero-point (klaylearn.com glossary "Weight-Only
 *    Quantisation", first FAQ answer and main body; multigrid.ai "Weight-Only
 *    Quantization Explained", section "What W4A16 actually names").
 *  - Groups of 32/64/128/256 weights each get their own scale (zhuai.tech
 *    "Quantization Is Not a Zip File", section 3 "The core idea: local
 *    structure, not global rounding", paragraph "Block locality").
 *  - Reconstruction of an asymmetric code is (q - zero_point) * scale
 *    (instagit.com "Comparison of Quantization Methods: INT8 vs GPTQ vs AWQ vs
 *    GGUF", section "Practical Code Examples", asymmetric example).
 *  - The layer output is dequantise-then-multiply (klaylearn.com glossary,
 *    main body: the kernel reconstructs 16-bit values of a tile and feeds a
 *    fused dequantise-and-multiply path).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * repository's design notes):
 *  - Layout: W is [N,K] (output column n, input channel k), y = x * W_hat^T.
 *    qweight[n][k/8] holds the code of k in bits 4*(k%8)..4*(k%8)+3 (low
 *    nibble first).  scales[n][g] is the FP16 scale of group g, row pitch
 *    ldS halves.  zeros[n][g/8] holds the 4-bit zero of group g in bits
 *    4*(g%8).., row pitch ldZ words.  Padding is written as zero.
 *  - Min-max range is widened to contain 0: lo = min(0, min w), hi = max(0,
 *    max w), so the zero point is a representable code.
 *  - scale = RNE_fp16( fp32(hi - lo) / 15 ) with IEEE single-precision
 *    subtraction and division; codes are computed against the stored FP16
 *    scale.  A scale that rounds to 0 is replaced by 1.0 with zero point 0.
 *  - zero = clamp(rne(-lo / s), 0, 15); q = clamp(rne(w / s) + zero, 0, 15),
 *    round-to-nearest-even, IEEE single-precision division.
 *  - W_hat = (float)(q - zero) * (float)s, which is exact in FP32.
 *  - y_ref[m][n] = sum_k (double)x[m][k] * (double)W_hat[n][k], accumulated in
 *    FP64 and left unrounded.
 *
 * Build: plain C99 with optional OpenMP (the parallel loops only split
 * independent output rows; each row's arithmetic order is fixed).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 / bfloat16 <-> binary32, written from the definitions.  */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);     /* (1.m) * 2^(e-15) */
    }
    return (float)(sign ? -v : v);
}

/* bfloat16: the top 16 bits of a binary32. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round a finite double to a binary format with `p` significand bits
 * (including the implicit one), minimum normal exponent `emin` and maximum
 * exponent `emax`, round-to-nearest, ties-to-even.  Returns the rounded value
 * as a double (or +-inf on overflow).  Used for binary16 (p=11, emin=-14,
 * emax=15) and bfloat16 (p=8, emin=-126, emax=127).
 */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1): exponent is e-1 */
    e -= 1;
    if (e < emin) e = emin;    /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, e - (p - 1));
    double m = nearbyint(a / quantum);           /* exact scaling, RNE */
    double r = m * quantum;
    /* overflow: the largest finite value is (2 - 2^(1-p)) * 2^emax */
    double maxfin = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (r > maxfin) r = INFINITY;
    return v < 0 ? -r : r;
}

uint16_t oracle_f32_to_f16(float f)
{
    if (isnan(f)) return 0x7E00;
    double r = round_to_format((double)f, 11, -14, 15);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14))                       /* subnormal */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    int e;
    frexp(a, &e);
    e -= 1;
    uint16_t mant = (uint16_t)(a / ldexp(1.0, e - 10) - 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | mant;
}

uint16_t oracle_f64_to_bf16(double d)
{
    if (isnan(d)) return 0x7FC0;
    double r = round_to_format(d, 8, -126, 127);
    float f = (float)r;                            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_bf16(float f) { return oracle_f64_to_bf16((double)f); }

/* ------------------------------------------------------------------------ */
/* Layout of the packed format.                                              */
/* ------------------------------------------------------------------------ */

static int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

/* uint32 words per row of qweight: 8 codes per word. */
int64_t oracle_qweight_ld(int64_t K) { return K / 8; }
/* halves per row of scales: K/G rounded up to 8 halves (16-byte pitch). */
int64_t oracle_scales_ld(int64_t K, int64_t G) { return round_up(K / G, 8); }
/* uint32 words per row of zeros: ceil(K/G / 8) rounded up to 4 words. */
int64_t oracle_zeros_ld(int64_t K, int64_t G) { return round_up((K / G + 7) / 8, 4); }

static int64_t clamp_i64(int64_t v, int64_t lo, int64_t hi)
{
    return v < lo ? lo : (v > hi ? hi : v);
}

/* ------------------------------------------------------------------------ */
/* Quantiser (packer): asymmetric min-max per group of G input channels.     */
/* ------------------------------------------------------------------------ */

/*
 * Quantise one group of G FP32 weights.  Writes the FP16 scale bits, the zero
 * point and G codes.  Follows the textbook asymmetric scheme: range -> scale,
 * zero point from the minimum, codes = round(w / scale) + zero, clamped to the
 * 4-bit grid [0, 15].
 */
void oracle_quantize_group(const float* w, int64_t G, uint16_t* scale_bits, int* zero, uint8_t* codes)
{
    float lo = 0.0f, hi = 0.0f;                    /* range widened to hold 0 */
    for (int64_t i = 0; i < G; ++i) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    volatile float range = hi - lo;                /* IEEE binary32 subtraction */
    volatile float s32 = range / 15.0f;            /* IEEE binary32 division */
    uint16_t sb = oracle_f32_to_f16(s32);
    float s = oracle_f16_to_f32(sb);
    int z;
    if (s == 0.0f) {                               /* degenerate group */
        sb = 0x3C00;                               /* 1.0 */
        s = 1.0f;
        z = 0;
    } else {
        volatile float t = -lo / s;
        z = (int)clamp_i64((int64_t)nearbyintf(t), 0, 15);
    }
    for (int64_t i = 0; i < G; ++i) {
        volatile float t = w[i] / s;
        int64_t q = (int64_t)nearbyintf(t) + z;
        codes[i] = (uint8_t)clamp_i64(q, 0, 15);
    }
    *scale_bits = sb;
    *zero = z;
}

/*
 * Pack an [N,K] FP16 weight (bits) into qweight [N, K/8], scales [N, ldS],
 * zeros [N, ldZ].  Output buffers are fully written, padding included.
 * Returns 0 on success, -1 on bad arguments.
 */
int oracle_pack(const uint16_t* w_f16, int64_t N, int64_t K, int64_t G,
                uint32_t* qweight, uint16_t* scales, uint32_t* zeros, int nthreads)
{
    if (N <= 0 || K <= 0 || G <= 0 || G > 256 || K % G != 0 || G % 8 != 0) return -1;
    const int64_t ldq = oracle_qweight_ld(K);
    const int64_t lds = oracle_scales_ld(K, G);
    const int64_t ldz = oracle_zeros_ld(K, G);
    const int64_t ngroups = K / G;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        float wf[256];
        uint8_t codes[256];
        uint32_t* qrow = qweight + n * ldq;
        uint16_t* srow = scales + n * lds;
        uint32_t* zrow = zeros + n * ldz;
        for (int64_t i = 0; i < ldq; ++i) qrow[i] = 0;
        for (int64_t i = 0; i < lds; ++i) srow[i] = 0;
        for (int64_t i = 0; i < ldz; ++i) zrow[i] = 0;
        for (int64_t g = 0; g < ngroups; ++g) {
            for (int64_t i = 0; i < G; ++i) wf[i] = oracle_f16_to_f32(w_f16[n * K + g * G + i]);
            uint16_t sb;
            int z;
            oracle_quantize_group(wf, G, &sb, &z, codes);
            srow[g] = sb;
            zrow[g / 8] |= (uint32_t)z << (4 * (g % 8));
            for (int64_t i = 0; i < G; ++i) {
                int64_t k = g * G + i;
                qrow[k / 8] |= (uint32_t)codes[i] << (4 * (k % 8));
            }
        }
    }
    (void)nthreads;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Unpack and dequantise.                                                    */
/* ------------------------------------------------------------------------ */

int oracle_code(const uint32_t* qweight, int64_t K, int64_t n, int64_t k)
{
    return (int)((qweight[n * oracle_qweight_ld(K) + k / 8] >> (4 * (k % 8))) & 0xF);
}

int oracle_zero(const uint32_t* zeros, int64_t K, int64_t G, int64_t n, int64_t g)
{
    return (int)((zeros[n * oracle_zeros_ld(K, G) + g / 8] >> (4 * (g % 8))) & 0xF);
}

float oracle_scale(const uint16_t* scales, int64_t K, int64_t G, int64_t n, int64_t g)
{
    return oracle_f16_to_f32(scales[n * oracle_scales_ld(K, G) + g]);
}

/* W_hat[n][k] = (q - z) * s in FP32 (exact: at most 15 significant bits). */
float oracle_dequant_one(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                         int64_t K, int64_t G, int64_t n, int64_t k)
{
    int64_t g = k / G;
    int q = oracle_code(qweight, K, n, k);
    int z = oracle_zero(zeros, K, G, n, g);
    float s = oracle_scale(scales, K, G, n, g);
    return (float)(q - z) * s;
}

/* Full dequantisation to an FP32 [N,K] matrix. */
void oracle_dequant(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                    int64_t N, int64_t K, int64_t G, float* w_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w_out[n * K + k] = oracle_dequant_one(qweight, scales, zeros, K, G, n, k);
    (void)nthreads;
}

/* ------------------------------------------------------------------------ */
/* The layer: y_ref = x * W_hat^T in FP64.                                   */
/* ------------------------------------------------------------------------ */

/* One output element, the plain definition. */
double oracle_linear_one(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                         const uint32_t* zeros, int64_t K, int64_t G, int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]);
        double wv = (double)oracle_dequant_one(qweight, scales, zeros, K, G, n, k);
        acc += xv * wv;
    }
    return acc;
}

/*
 * y_ref [M,N] (FP64) for all outputs: every element is the plain definition
 * of oracle_linear_one (products summed over k in increasing order).
 */
void oracle_linear(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                   const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int64_t G,
                   double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            y_out[m * N + n] = oracle_linear_one(x_bf16, qweight, scales, zeros, K, G, m, n);
    (void)nthreads;
}

/* Selected outputs only: y_out[i] = y_ref[ms[i]][ns[i]]. */
void oracle_linear_sampled(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                           const uint32_t* zeros, int64_t K, int64_t G, const int64_t* ms,
                           const int64_t* ns, int64_t count, double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < count; ++i)
        y_out[i] = oracle_linear_one(x_bf16, qweight, scales, zeros, K, G, ms[i], ns[i]);
    (void)nthreads;
}

/*
 * The layer with a per-input-channel activation scale, the deployed form of
 * activation-aware weight quantisation: salient input channels have their
 * weights scaled up before quantisation and the activations scaled down by
 * the same factor, so the layer itself stays an ordinary groupwise INT4
 * dequantise-then-multiply (instagit.com "Comparison of Quantization Methods:
 * INT8 vs GPTQ vs AWQ vs GGUF", section "AWQ: Activation-Aware Weight
 * Quantization"; klaylearn.com glossary, FAQ "What is the difference between
 * AWQ and GPTQ?").  x_scale[k] is the factor applied to input channel k:
 *   y_ref[m][n] = sum_k (double)x[m][k] * (double)x_scale[k] * (double)W_hat[n][k],
 * accumulated in FP64 in increasing k and left unrounded.
 */
double oracle_linear_xs_one(const uint16_t* x_bf16, const float* x_scale, const uint32_t* qweight,
                            const uint16_t* scales, const uint32_t* zeros, int64_t K, int64_t G, int64_t m,
                            int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]) * (double)x_scale[k];
        double wv = (double)oracle_dequant_one(qweight, scales, zeros, K, G, n, k);
        acc += xv * wv;
    }
    return acc;
}

void oracle_linear_xs(const uint16_t* x_bf16, const float* x_scale, const uint32_t* qweight,
                      const uint16_t* scales, const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int64_t G,
                      double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            y_out[m * N + n] = oracle_linear_xs_one(x_bf16, x_scale, qweight, scales, zeros, K, G, m, n);
    (void)nthreads;
}

/* ------------------------------------------------------------------------ */
/* The 8-bit variant (W8A16).                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Weight-only quantisation stores the weights as INT8 or INT4 and leaves the
 * activations in 16-bit (klaylearn.com glossary "Weight-Only Quantisation",
 * first FAQ answer and main body).  The 8-bit quantiser here is the 4-bit one
 * with 255 steps:
 *   lo = min(0, min w), hi = max(0, max w)
 *   s8 = RNE_fp16( fp32(hi - lo) / 255 ); s8 == 0 -> s8 = 1, z8 = 0
 *   z8 = clamp(rne(-lo / s8), 0, 255),  q8 = clamp(rne(w / s8) + z8, 0, 255)
 * Storage (a reading; the pages give none): an 8-bit code is kept as two 4-bit
 * planes of a 4-bit layer with 2K input channels.  Row n holds the K high
 * nibbles q8 >> 4 (channels 0..K-1) followed by the K low nibbles q8 & 15
 * (channels K..2K-1) in the 4-bit layout; its scales are the K/G hi-plane
 * scales 16*s8 followed by the K/G lo-plane scales s8, its zeros z8 >> 4 then
 * z8 & 15.  8 bits per weight; row pitches those of the 2K-channel 4-bit layer.
 */
void oracle_quantize_group8(const float* w, int64_t G, uint16_t* scale_bits, int* zero, int* codes)
{
    float lo = 0.0f, hi = 0.0f;
    for (int64_t i = 0; i < G; ++i) {
        if (w[i] < lo) lo = w[i];
        if (w[i] > hi) hi = w[i];
    }
    volatile float range = hi - lo;
    volatile float s32 = range / 255.0f;
    uint16_t sb = oracle_f32_to_f16(s32);
    float s = oracle_f16_to_f32(sb);
    int z;
    if (s == 0.0f) {
        sb = 0x3C00;
        s = 1.0f;
        z = 0;
    } else {
        volatile float t = -lo / s;
        z = (int)clamp_i64((int64_t)nearbyintf(t), 0, 255);
    }
    for (int64_t i = 0; i < G; ++i) {
        volatile float t = w[i] / s;
        int64_t q = (int64_t)nearbyintf(t) + z;
        codes[i] = (int)clamp_i64(q, 0, 255);
    }
    *scale_bits = sb;
    *zero = z;
}

int oracle_pack8(const uint16_t* w_f16, int64_t N, int64_t K, int64_t G,
                 uint32_t* qweight, uint16_t* scales, uint32_t* zeros, int nthreads)
{
    if (N <= 0 || K <= 0 || G <= 0 || G > 256 || K % G != 0 || G % 8 != 0) return -1;
    const int64_t K2 = 2 * K;
    const int64_t ldq = oracle_qweight_ld(K2);
    const int64_t lds = oracle_scales_ld(K2, G);
    const int64_t ldz = oracle_zeros_ld(K2, G);
    const int64_t ngroups = K / G;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        float wf[256];
        int codes[256];
        uint32_t* qrow = qweight + n * ldq;
        uint16_t* srow = scales + n * lds;
        uint32_t* zrow = zeros + n * ldz;
        for (int64_t i = 0; i < ldq; ++i) qrow[i] = 0;
        for (int64_t i = 0; i < lds; ++i) srow[i] = 0;
        for (int64_t i = 0; i < ldz; ++i) zrow[i] = 0;
        for (int64_t g = 0; g < ngroups; ++g) {
            for (int64_t i = 0; i < G; ++i) wf[i] = oracle_f16_to_f32(w_f16[n * K + g * G + i]);
            uint16_t sb;
            int z;
            oracle_quantize_group8(wf, G, &sb, &z, codes);
            srow[g] = oracle_f32_to_f16(16.0f * oracle_f16_to_f32(sb));   /* exact: a power-of-two scaling */
            srow[ngroups + g] = sb;
            zrow[g / 8] |= (uint32_t)(z >> 4) << (4 * (g % 8));
            zrow[(ngroups + g) / 8] |= (uint32_t)(z & 15) << (4 * ((ngroups + g) % 8));
            for (int64_t i = 0; i < G; ++i) {
                int64_t k = g * G + i;
                qrow[k / 8] |= (uint32_t)(codes[i] >> 4) << (4 * (k % 8));
                qrow[(K + k) / 8] |= (uint32_t)(codes[i] & 15) << (4 * ((K + k) % 8));
            }
        }
    }
    (void)nthreads;
    return 0;
}

/* The 8-bit code, zero point and scale of weight (n, k) read back from the planes. */
static int oracle_code8(const uint32_t* qweight, int64_t K, int64_t n, int64_t k)
{
    return 16 * oracle_code(qweight, 2 * K, n, k) + oracle_code(qweight, 2 * K, n, K + k);
}
static int oracle_zero8(const uint32_t* zeros, int64_t K, int64_t G, int64_t n, int64_t g)
{
    return 16 * oracle_zero(zeros, 2 * K, G, n, g) + oracle_zero(zeros, 2 * K, G, n, K / G + g);
}

/* W_hat8 = (q8 - z8) * s8, exact in FP32 (at most 9 + 11 significant bits). */
float oracle_dequant8_one(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                          int64_t K, int64_t G, int64_t n, int64_t k)
{
    int64_t g = k / G;
    int q = oracle_code8(qweight, K, n, k);
    int z = oracle_zero8(zeros, K, G, n, g);
    float s = oracle_scale(scales, 2 * K, G, n, K / G + g);
    return (float)(q - z) * s;
}

void oracle_dequant8(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                     int64_t N, int64_t K, int64_t G, float* w_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w_out[n * K + k] = oracle_dequant8_one(qweight, scales, zeros, K, G, n, k);
    (void)nthreads;
}

/* y_ref[m][n] = sum_k (double)x[m][k] * (double)W_hat8[n][k], FP64 in increasing k, unrounded. */
void oracle_linear8(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                    const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int64_t G, double* y_out,
                    int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]);
                double wv = (double)oracle_dequant8_one(qweight, scales, zeros, K, G, n, k);
                acc += xv * wv;
            }
            y_out[m * N + n] = acc;
        }
    (void)nthreads;
}

/* ------------------------------------------------------------------------ */
/* The 8-bit variant in the word layout: four codes per 32-bit word.           */
/* ------------------------------------------------------------------------ */

/*
 * The pages name INT8 beside INT4 as the weight width of weight-only
 * quantisation with 16-bit activations (klaylearn.com glossary "Weight-Only
 * Quantisation", first FAQ answer) and give no 8-bit layout.  Reading: the
 * same groups and the same 255-step quantiser as oracle_quantize_group8, with
 * the metadata of the 4-bit layout widened to 8 bits:
 *   qweight [N, K/4]          code of (n, k) in bits 8*(k%4) .. 8*(k%4)+7 of
 *                             word k/4 (low byte first)
 *   scales  [N, ldS(K, G)]    FP16 scale of group g, as the 4-bit layout
 *   zeros   [N, ldZ8(K, G)]   8-bit zero point of group g in bits 8*(g%4) ..
 *                             of word g/4; ldZ8 = ceil(K/G / 4) rounded up to
 *                             a multiple of 4 words (16-byte rows)
 *   W_hat = (q - z) * s, exact in FP32.
 * Padding words and halves are zero.
 */
int64_t oracle_zeros8w_ld(int64_t K, int64_t G) { return round_up((K / G + 3) / 4, 4); }

int oracle_pack8w(const uint16_t* w_f16, int64_t N, int64_t K, int64_t G,
                  uint32_t* qweight, uint16_t* scales, uint32_t* zeros, int nthreads)
{
    if (N <= 0 || K <= 0 || G <= 0 || G > 256 || K % G != 0 || G % 8 != 0) return -1;
    const int64_t ldq = K / 4;
    const int64_t lds = oracle_scales_ld(K, G);
    const int64_t ldz = oracle_zeros8w_ld(K, G);
    const int64_t ngroups = K / G;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        float wf[256];
        int codes[256];
        uint32_t* qrow = qweight + n * ldq;
        uint16_t* srow = scales + n * lds;
        uint32_t* zrow = zeros + n * ldz;
        for (int64_t i = 0; i < ldq; ++i) qrow[i] = 0;
        for (int64_t i = 0; i < lds; ++i) srow[i] = 0;
        for (int64_t i = 0; i < ldz; ++i) zrow[i] = 0;
        for (int64_t g = 0; g < ngroups; ++g) {
            for (int64_t i = 0; i < G; ++i) wf[i] = oracle_f16_to_f32(w_f16[n * K + g * G + i]);
            uint16_t sb;
            int z;
            oracle_quantize_group8(wf, G, &sb, &z, codes);
            srow[g] = sb;
            zrow[g / 4] |= (uint32_t)z << (8 * (g % 4));
            for (int64_t i = 0; i < G; ++i) {
                const int64_t k = g * G + i;
                qrow[k / 4] |= (uint32_t)codes[i] << (8 * (k % 4));
            }
        }
    }
    (void)nthreads;
    return 0;
}

/* W_hat = (q - z) * s of weight (n, k) in the word layout, exact in FP32. */
float oracle_dequant8w_one(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                           int64_t K, int64_t G, int64_t n, int64_t k)
{
    const int64_t g = k / G;
    const int q = (int)((qweight[n * (K / 4) + k / 4] >> (8 * (k % 4))) & 0xFFu);
    const int z = (int)((zeros[n * oracle_zeros8w_ld(K, G) + g / 4] >> (8 * (g % 4))) & 0xFFu);
    const float s = oracle_f16_to_f32(scales[n * oracle_scales_ld(K, G) + g]);
    return (float)(q - z) * s;
}

void oracle_dequant8w(const uint32_t* qweight, const uint16_t* scales, const uint32_t* zeros,
                      int64_t N, int64_t K, int64_t G, float* w_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w_out[n * K + k] = oracle_dequant8w_one(qweight, scales, zeros, K, G, n, k);
    (void)nthreads;
}

/* y_ref[m][n] = sum_k (double)x[m][k] * (double)W_hat[n][k], FP64 in increasing k, unrounded. */
double oracle_linear8w_one(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                           const uint32_t* zeros, int64_t K, int64_t G, int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]);
        double wv = (double)oracle_dequant8w_one(qweight, scales, zeros, K, G, n, k);
        acc += xv * wv;
    }
    return acc;
}

void oracle_linear8w(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                     const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int64_t G, double* y_out,
                     int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) y_out[m * N + n] = oracle_linear8w_one(x_bf16, qweight, scales, zeros, K, G, m, n);
    (void)nthreads;
}

void oracle_linear8w_sampled(const uint16_t* x_bf16, const uint32_t* qweight, const uint16_t* scales,
                             const uint32_t* zeros, int64_t K, int64_t G, const int64_t* ms, const int64_t* ns,
                             int64_t count, double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < count; ++i)
        y_out[i] = oracle_linear8w_one(x_bf16, qweight, scales, zeros, K, G, ms[i], ns[i]);
    (void)nthreads;
}

/* ------------------------------------------------------------------------ */
/* The super-block variant (Q4_K-style K-quant).                              */
/* ------------------------------------------------------------------------ */

/*
 * K-quants keep 4-bit codes in 256-weight super-blocks whose sub-blocks carry
 * their own scale and minimum, and those scales are themselves quantised
 * against per-super-block factors (zhuai.tech "Quantization Is Not a Zip
 * File", section 3 "The core idea: local structure, not global rounding",
 * table "How to read common GGUF quantization names", K-quants row and the
 * note on hierarchical K-quant scales; section 2 "Moving fewer bytes can make
 * decode faster" on packed Q4_K decode dot products).
 *
 * Readings where the pages are silent:
 *  - A super-block is 256 consecutive input channels of one output row, cut
 *    into 8 sub-blocks of 32.  Sub-block j reconstructs as
 *        W_hat = a'_j * q - b'_j,   a'_j = d * sc_j,   b'_j = dmin * m_j,
 *    with q in [0, 15], 6-bit codes sc_j, m_j in [0, 63], and FP16 factors
 *    d, dmin per super-block.  a'_j and b'_j are exact in FP32 (11 + 6
 *    significant bits), so is a'_j * q (17 + 4); W_hat rounds once, at the
 *    FP32 subtraction.
 *  - Quantiser (min-max, no search), all decisions in IEEE binary32:
 *        lo_j = min(0, min w), hi_j = max(0, max w)   (range holds 0)
 *        a_j = (hi_j - lo_j) / 15,  b_j = -lo_j
 *        d = RNE_fp16(max_j a_j / 63),  dmin = RNE_fp16(max_j b_j / 63)
 *        d == 0 -> d = 1.0;  sc_j = clamp(rne(a_j / d), 0, 63)
 *        dmin == 0 -> m_j = 0, else m_j = clamp(rne(b_j / dmin), 0, 63)
 *        q = a'_j > 0 ? clamp(rne((w + b'_j) / a'_j), 0, 15) : 0
 *  - Storage: qweight as the 4-bit layer ([N, K/8] words, low nibble first);
 *    meta [N, K/256 * 4] words, one 16-byte record per super-block:
 *        word 0: d bits (low half), dmin bits (high half)
 *        word 1: sc_j & 15 at bits 4j..4j+3
 *        word 2: m_j & 15 at bits 4j..4j+3
 *        word 3: sc_j >> 4 at bits 2j..2j+1, m_j >> 4 at bits 16+2j..17+2j
 *    4.5 bits per weight.  K must be a multiple of 256.
 */
int64_t oracle_q4k_meta_ld(int64_t K) { return K / 256 * 4; }

/* Quantise one super-block of 256 FP32 weights: FP16 bits of d and dmin, the
 * 8 sub-block codes sc[] and m[], and 256 codes q[]. */
void oracle_q4k_quantize_superblock(const float* w, uint16_t* d_bits, uint16_t* dmin_bits, int* sc, int* m,
                                    uint8_t* q)
{
    float a[8], b[8], amax = 0.0f, bmax = 0.0f;
    for (int j = 0; j < 8; ++j) {
        float lo = 0.0f, hi = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float v = w[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        volatile float range = hi - lo;
        volatile float aj = range / 15.0f;
        a[j] = aj;
        b[j] = -lo;
        if (a[j] > amax) amax = a[j];
        if (b[j] > bmax) bmax = b[j];
    }
    volatile float dq = amax / 63.0f, dmq = bmax / 63.0f;
    uint16_t db = oracle_f32_to_f16(dq), dmb = oracle_f32_to_f16(dmq);
    float d = oracle_f16_to_f32(db), dmin = oracle_f16_to_f32(dmb);
    if (d == 0.0f) {
        db = 0x3C00;
        d = 1.0f;
    }
    for (int j = 0; j < 8; ++j) {
        volatile float ts = a[j] / d;
        sc[j] = (int)clamp_i64((int64_t)nearbyintf(ts), 0, 63);
        if (dmin == 0.0f) {
            m[j] = 0;
        } else {
            volatile float tm = b[j] / dmin;
            m[j] = (int)clamp_i64((int64_t)nearbyintf(tm), 0, 63);
        }
        float ap = d * (float)sc[j], bp = dmin * (float)m[j];      /* exact products */
        for (int i = 0; i < 32; ++i) {
            if (ap > 0.0f) {
                volatile float sum = w[32 * j + i] + bp;
                volatile float t = sum / ap;
                q[32 * j + i] = (uint8_t)clamp_i64((int64_t)nearbyintf(t), 0, 15);
            } else {
                q[32 * j + i] = 0;
            }
        }
    }
    *d_bits = db;
    *dmin_bits = dmb;
}

/* Pack an [N,K] FP16 weight into qweight [N, K/8] and meta [N, K/256*4]. */
int oracle_q4k_pack(const uint16_t* w_f16, int64_t N, int64_t K, uint32_t* qweight, uint32_t* meta, int nthreads)
{
    if (N <= 0 || K <= 0 || K % 256 != 0) return -1;
    const int64_t ldq = oracle_qweight_ld(K);
    const int64_t ldm = oracle_q4k_meta_ld(K);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        float wf[256];
        uint8_t codes[256];
        int sc[8], m[8];
        uint32_t* qrow = qweight + n * ldq;
        uint32_t* mrow = meta + n * ldm;
        for (int64_t i = 0; i < ldq; ++i) qrow[i] = 0;
        for (int64_t i = 0; i < ldm; ++i) mrow[i] = 0;
        for (int64_t sb = 0; sb < K / 256; ++sb) {
            for (int i = 0; i < 256; ++i) wf[i] = oracle_f16_to_f32(w_f16[n * K + sb * 256 + i]);
            uint16_t db, dmb;
            oracle_q4k_quantize_superblock(wf, &db, &dmb, sc, m, codes);
            uint32_t* rec = mrow + sb * 4;
            rec[0] = (uint32_t)db | ((uint32_t)dmb << 16);
            for (int j = 0; j < 8; ++j) {
                rec[1] |= (uint32_t)(sc[j] & 15) << (4 * j);
                rec[2] |= (uint32_t)(m[j] & 15) << (4 * j);
                rec[3] |= (uint32_t)(sc[j] >> 4) << (2 * j);
                rec[3] |= (uint32_t)(m[j] >> 4) << (16 + 2 * j);
            }
            for (int i = 0; i < 256; ++i) {
                int64_t k = sb * 256 + i;
                qrow[k / 8] |= (uint32_t)codes[i] << (4 * (k % 8));
            }
        }
    }
    (void)nthreads;
    return 0;
}

/* The 6-bit codes of sub-block j and the factors of super-block sb, read back from the record. */
void oracle_q4k_record(const uint32_t* meta, int64_t K, int64_t n, int64_t sb, float* d, float* dmin, int* sc,
                       int* m)
{
    const uint32_t* rec = meta + n * oracle_q4k_meta_ld(K) + sb * 4;
    *d = oracle_f16_to_f32((uint16_t)(rec[0] & 0xFFFF));
    *dmin = oracle_f16_to_f32((uint16_t)(rec[0] >> 16));
    for (int j = 0; j < 8; ++j) {
        sc[j] = (int)(((rec[1] >> (4 * j)) & 15) | (((rec[3] >> (2 * j)) & 3) << 4));
        m[j] = (int)(((rec[2] >> (4 * j)) & 15) | (((rec[3] >> (16 + 2 * j)) & 3) << 4));
    }
}

/* W_hat[n][k] = (d * sc_j) * q - dmin * m_j in FP32 (the two products exact, one rounding). */
float oracle_q4k_dequant_one(const uint32_t* qweight, const uint32_t* meta, int64_t K, int64_t n, int64_t k)
{
    float d, dmin;
    int sc[8], m[8];
    oracle_q4k_record(meta, K, n, k / 256, &d, &dmin, sc, m);
    const int j = (int)((k % 256) / 32);
    const int q = oracle_code(qweight, K, n, k);
    volatile float ap = d * (float)sc[j];
    volatile float bp = dmin * (float)m[j];
    volatile float t = ap * (float)q;                  /* exact: at most 17 + 4 significant bits */
    return t - bp;
}

void oracle_q4k_dequant(const uint32_t* qweight, const uint32_t* meta, int64_t N, int64_t K, float* w_out,
                        int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) w_out[n * K + k] = oracle_q4k_dequant_one(qweight, meta, K, n, k);
    (void)nthreads;
}

/* y_ref[m][n] = sum_k (double)x[m][k] * (double)W_hat[n][k], FP64 in increasing k, unrounded. */
double oracle_q4k_linear_one(const uint16_t* x_bf16, const uint32_t* qweight, const uint32_t* meta, int64_t K,
                             int64_t m, int64_t n)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]);
        double wv = (double)oracle_q4k_dequant_one(qweight, meta, K, n, k);
        acc += xv * wv;
    }
    return acc;
}

void oracle_q4k_linear(const uint16_t* x_bf16, const uint32_t* qweight, const uint32_t* meta, int64_t M,
                       int64_t N, int64_t K, double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) y_out[m * N + n] = oracle_q4k_linear_one(x_bf16, qweight, meta, K, m, n);
    (void)nthreads;
}

void oracle_q4k_linear_sampled(const uint16_t* x_bf16, const uint32_t* qweight, const uint32_t* meta, int64_t K,
                               const int64_t* ms, const int64_t* ns, int64_t count, double* y_out, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < count; ++i) y_out[i] = oracle_q4k_linear_one(x_bf16, qweight, meta, K, ms[i], ns[i]);
    (void)nthreads;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
