/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the weight-only
 * quantized GEMV formats.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or constant
 * with the CUDA library, and the CUDA library never loads it.
 *
 * Every dot product accumulates in double and is returned in double.  With the
 * workloads' value ranges each product term is exact in double (int4 x f32
 * scale x f32/bf16 activation, e4m3 x f32 x bf16, fp16-affine x bf16), so the
 * only rounding is the order of summation.  Each function cites the passage
 * of the page it follows:
 *
 *   [colibri #457]  "metal: grouped-int4 (fmt=4) GEMV support", sections 3-5, 7, 11
 *   [colibri #528]  "fmt=7: fp8-e4m3-b128 passthrough weight format", Design
 *                   (f32 block scales, and the UE8M0 scale encoding it names)
 *   [hipfire MQ4V2] "MQ4 V2" docs, sections 1b, 1c, 1e, 2, 3, 4, 9
 *   [strata Q2_0]   strata review, "convert_k256_q2_0.cpp vs ref_quant.cpp" (2.5)
 *
 * No function here blocks, fuses or reorders beyond what its definition
 * states; loops run in the order the definition reads.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar number formats                                                    */
/* ------------------------------------------------------------------------ */

/* OCP 8-bit floating point, E4M3 "FN" variant ([colibri #528] Design: the
 * decode table is exact OCP E4M3-FN; the only NaN codes have every exponent
 * bit and every mantissa bit set; an all-ones exponent is NOT infinity).
 *   sign s = bit 7, exponent e = bits 6..3 (bias 7), mantissa m = bits 2..0
 *   e == 15 && m == 7 : NaN (codes 0x7F and 0xFF)
 *   e == 0            : subnormal, (-1)^s * 2^(1-7) * (m/8)
 *   otherwise         : normal,    (-1)^s * 2^(e-7) * (1 + m/8)            */
double oracle_e4m3_value(uint8_t code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* IEEE 754 binary16: sign bit 15, exponent bits 14..10 (bias 15), fraction
 * bits 9..0.  Used for the MQ4-V2 header ([hipfire MQ4V2] section 2).        */
double oracle_f16_value(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 31)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return s ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even (IEEE 754 default).
 * Written from the definition: find the binade, scale the value so that one
 * unit in the last place of the target is 1.0, round to the nearest integer
 * with ties going to even, and re-assemble.  All the double arithmetic here
 * is exact (power-of-two scaling of a value with at most 24 significant
 * bits), so rint() does the only rounding, in the default rounding mode.    */
uint16_t oracle_f16_from_f32(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00u);
    if (a >= 65520.0)            /* halfway between 65504 and 2^16 and above */
        return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {   /* subnormal range: ulp is 2^-24 */
        double q = rint(a / ldexp(1.0, -24));
        /* q == 1024 rounds up into the smallest normal; the bit pattern
         * 0x0400 is exactly that, so no special case is needed.            */
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    (void)frexp(a, &e2);         /* a = fr * 2^e2 with fr in [0.5, 1) */
    int e = e2 - 1;              /* a in [2^e, 2^(e+1)) */
    double frac = rint((a / ldexp(1.0, e) - 1.0) * 1024.0);
    if (frac >= 1024.0) {        /* rounded up to the next binade */
        frac = 0.0;
        e += 1;
    }
    if (e + 15 >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)frac);
}

/* bfloat16 is the upper half of a binary32: widening is exact. */
double oracle_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* fmt=4: grouped int4 ([colibri #457] sections 3, 11)                       */
/*   w: O rows of rb = (I+1)/2 bytes; element i of row o sits in byte i/2,   */
/*      the low nibble for even i, the high nibble for odd i; the stored     */
/*      nibble n means the integer n - 8.                                    */
/*   scales: f32 [O, ng], ng = ceil(I/gs); element i uses scale[o*ng + i/gs] */
/*   y[s,o] = sum_i (n(o,i) - 8) * scale[o, i/gs] * x[s,i]                   */
/* The scale multiplies every term (per group, before summing across         */
/* groups); it is never applied once to the finished row sum.                */
/* ------------------------------------------------------------------------ */

static int i4g_value(const uint8_t *w, size_t rb, int o, int i)
{
    uint8_t byte = w[(size_t)o * rb + (size_t)(i / 2)];
    int nib = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return nib - 8;
}

/* y and mag are double [S, O].  mag[s,o] = sum_i |term_i| is the magnitude
 * that the relative tolerance is measured against ([colibri #457] section 5:
 * per-element |delta| / sum |x_i * (n-8) * scale|).                         */
void oracle_qgemv_i4g(double *y, double *mag, const float *x, const uint8_t *w,
                      const float *scales, int S, int I, int O, int gs)
{
    size_t rb = ((size_t)I + 1) / 2;
    size_t ng = ((size_t)I + (size_t)gs - 1) / (size_t)gs;
    for (int s = 0; s < S; ++s) {
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (int i = 0; i < I; ++i) {
                double q = (double)i4g_value(w, rb, o, i);
                double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];
                double t = q * sc * (double)x[(size_t)s * I + i];
                acc += t;
                m += fabs(t);
            }
            y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
    }
}

/* Batched prefill for fmt=4: the same sum with bf16 activations X[M, I]
 * ([colibri #457] section 4: the large-batch GEMM path computes the same
 * grouped product as the GEMV).                                             */
void oracle_qgemm_i4g(double *Y, double *mag, const uint16_t *X, const uint8_t *w,
                      const float *scales, int M, int I, int O, int gs)
{
    size_t rb = ((size_t)I + 1) / 2;
    size_t ng = ((size_t)I + (size_t)gs - 1) / (size_t)gs;
    for (int s = 0; s < M; ++s) {
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (int i = 0; i < I; ++i) {
                double q = (double)i4g_value(w, rb, o, i);
                double sc = (double)scales[(size_t)o * ng + (size_t)(i / gs)];
                double t = q * sc * oracle_bf16_value(X[(size_t)s * I + i]);
                acc += t;
                m += fabs(t);
            }
            Y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
    }
}

/* Symmetric per-group int4 quantizer used to build fmt=4 weights.
 *   scale_g = max_{i in g} |w_i| / 7          (binary32 division)
 *   q_i     = clamp(rint(w_i / scale_g), -8, 7), stored as q_i + 8
 *   an all-zero group gets scale 0 and every nibble 8 (value 0).
 * An odd I leaves the high nibble of each row's last byte unused; it is
 * written as 8 (value 0).  The rounding is binary32 round-to-nearest-even
 * on both the division and rint, so any implementation taking the same
 * binary32 steps produces identical bytes.                                  */
void oracle_quantize_i4g(uint8_t *wq, float *scales, const float *w, int O, int I, int gs)
{
    size_t rb = ((size_t)I + 1) / 2;
    size_t ng = ((size_t)I + (size_t)gs - 1) / (size_t)gs;
    for (int o = 0; o < O; ++o) {
        memset(wq + (size_t)o * rb, 0x88, rb);
        for (size_t g = 0; g < ng; ++g) {
            int i0 = (int)(g * (size_t)gs);
            int i1 = i0 + gs < I ? i0 + gs : I;
            float amax = 0.0f;
            for (int i = i0; i < i1; ++i) {
                float a = fabsf(w[(size_t)o * I + i]);
                if (a > amax)
                    amax = a;
            }
            volatile float sc = amax / 7.0f;
            scales[(size_t)o * ng + g] = sc;
            for (int i = i0; i < i1; ++i) {
                int q = 0;
                if (sc != 0.0f) {
                    volatile float r = w[(size_t)o * I + i] / sc;
                    float qr = rintf(r);
                    if (qr < -8.0f) qr = -8.0f;
                    if (qr > 7.0f) qr = 7.0f;
                    q = (int)qr;
                }
                uint8_t nib = (uint8_t)(q + 8);
                uint8_t *byte = wq + (size_t)o * rb + (size_t)(i / 2);
                if (i % 2 == 0)
                    *byte = (uint8_t)((*byte & 0xF0) | nib);
                else
                    *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* fmt=7: FP8-e4m3, 128x128 block scales ([colibri #528] Design)             */
/*   w: O*I e4m3 codes, row-major [O, I]                                     */
/*   scale_inv: f32, one per 128x128 block, ceil(O/128) x ceil(I/128),       */
/*              row-major block order                                        */
/*   W[o,i] = e4m3(w[o*I+i]) * scale_inv[(o/128)*ceil(I/128) + i/128]        */
/*   (multiply, not divide); partial edge blocks use the same indexing.      */
/*   A NaN weight makes its output row NaN through the sum.                  */
/* ------------------------------------------------------------------------ */
void oracle_qgemv_fp8b128(double *y, double *mag, const uint16_t *x, const uint8_t *w,
                          const float *scale_inv, int S, int I, int O)
{
    size_t nbi = ((size_t)I + 127) / 128;
    for (int s = 0; s < S; ++s) {
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (int i = 0; i < I; ++i) {
                double wv = oracle_e4m3_value(w[(size_t)o * I + i]);
                double sc = (double)scale_inv[(size_t)(o / 128) * nbi + (size_t)(i / 128)];
                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);
                acc += t;
                m += fabs(t);
            }
            y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q2_0 ([strata Q2_0]: the ggml Q2_0 codec the review checks)                */
/*                                                                           : 18 bytes per 64 weights, little-endian:                  */
/*     [0,2)   fp16 d                                                         */
/*     [2,18)  16 bytes of 2-bit codes; weight e of the block sits in byte    */
/*             2 + e/4 at bit 2*(e%4)                                         */
/*   w_e = (code_e - 1) * d   (the asymmetric grid {-1, 0, 1, 2} * d).        */
/*   Row o holds I/64 blocks back to back; I must be a multiple of 64.        */
/* ------------------------------------------------------------------------ */
double oracle_q2_0_weight(const uint8_t *block, int e)
{
    double d = oracle_f16_value((uint16_t)(block[0] | (block[1] << 8)));
    int code = (block[2 + e / 4] >> (2 * (e % 4))) & 3;
    return (double)(code - 1) * d;
}

void oracle_qgemv_q2_0(double *y, double *mag, const uint16_t *x, const uint8_t *blocks, int S, int I, int O)
{
    const size_t nb = (size_t)I / 64;
    for (int s = 0; s < S; ++s)
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (int i = 0; i < I; ++i) {
                double t = oracle_q2_0_weight(blocks + ((size_t)o * nb + (size_t)(i / 64)) * 18, i % 64) *
                           oracle_bf16_value(x[(size_t)s * I + i]);
                acc += t;
                m += fabs(t);
            }
            y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
}

/* Encoder (the same review, 2.5: "searches d in {0.5 ... 1.0} * amax (9
 * steps) for minimal SSE on the asymmetric {-1,0,1,2} grid ... the error is
 * evaluated with the unrounded d").  Reading: per block amax = max |w|
 * (binary32); for k = 0..8 the candidate d_k = amax * (0.5 + k/16) (binary32),
 * codes c = clamp(rint(w / d_k) + 1, 0, 3) (binary32 division and rint),
 * SSE = sum (w - (c - 1) d_k)^2 in double; the first candidate with the
 * smallest SSE wins; its codes are stored with fp16(d_k) (round to nearest
 * even).  An all-zero block stores d = 0 and codes 1.                        */
void oracle_encode_q2_0(uint8_t *blocks, const float *w, int O, int I)
{
    const size_t nb = (size_t)I / 64;
    for (int o = 0; o < O; ++o)
        for (size_t b = 0; b < nb; ++b) {
            const float *v = w + (size_t)o * I + b * 64;
            uint8_t *out = blocks + ((size_t)o * nb + b) * 18;
            float amax = 0.0f;
            for (int e = 0; e < 64; ++e)
                amax = fabsf(v[e]) > amax ? fabsf(v[e]) : amax;
            int best_code[64];
            float best_d = 0.0f;
            for (int e = 0; e < 64; ++e)
                best_code[e] = 1;
            if (amax > 0.0f) {
                double best_sse = INFINITY;
                for (int k = 0; k <= 8; ++k) {
                    volatile float frac = 0.5f + (float)k / 16.0f;
                    volatile float d = amax * frac;
                    int code[64];
                    double sse = 0.0;
                    for (int e = 0; e < 64; ++e) {
                        volatile float r = v[e] / d;
                        float q = rintf(r) + 1.0f;
                        int c = q < 0.0f ? 0 : q > 3.0f ? 3 : (int)q;
                        code[e] = c;
                        double err = (double)v[e] - (double)(c - 1) * (double)d;
                        sse += err * err;
                    }
                    if (sse < best_sse) {
                        best_sse = sse;
                        best_d = d;
                        for (int e = 0; e < 64; ++e)
                            best_code[e] = code[e];
                    }
                }
            }
            uint16_t d16 = oracle_f16_from_f32(best_d);
            out[0] = (uint8_t)(d16 & 0xFF);
            out[1] = (uint8_t)(d16 >> 8);
            for (int j = 0; j < 16; ++j)
                out[2 + j] = (uint8_t)(best_code[4 * j] | (best_code[4 * j + 1] << 2) | (best_code[4 * j + 2] << 4) |
                                       (best_code[4 * j + 3] << 6));
        }
}

/* ------------------------------------------------------------------------ */
/* fmt=7 with UE8M0 block scales ([colibri #528] Design: the scale encoding  */
/* is a declared property of the format; DeepSeek-V4 ships the same e4m3     */
/* geometry with one byte per 128x128 block holding a power-of-two exponent, */
/* dtype F8_E8M0).  The page gives no bias; the reading taken is the OCP MX  */
/* E8M0 type that name denotes: byte e means 2^(e - 127), e = 255 is NaN.    */
/*   W[o,i] = e4m3(w[o*I+i]) * 2^(scale_e8m0[(o/128)*ceil(I/128) + i/128] - 127) */
/* ------------------------------------------------------------------------ */
double oracle_e8m0_value(uint8_t e)
{
    if (e == 255)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

void oracle_qgemv_fp8ue8m0(double *y, double *mag, const uint16_t *x, const uint8_t *w,
                           const uint8_t *scale_e8m0, int S, int I, int O)
{
    size_t nbi = ((size_t)I + 127) / 128;
    for (int s = 0; s < S; ++s) {
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (int i = 0; i < I; ++i) {
                double wv = oracle_e4m3_value(w[(size_t)o * I + i]);
                double sc = oracle_e8m0_value(scale_e8m0[(size_t)(o / 128) * nbi + (size_t)(i / 128)]);
                double t = wv * sc * oracle_bf16_value(x[(size_t)s * I + i]);
                acc += t;
                m += fabs(t);
            }
            y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MQ4-V2 (qt=44) ([hipfire MQ4V2] sections 2 and 4)                         */
/*   136 bytes per 256 weights, little-endian:                               */
/*     [0,4)   dword hA: low 16 bits fp16 scale, high 16 bits fp16 zero,     */
/*             for weights 0..127 of the block (half 0)                      */
/*     [4,8)   dword hB: the same for weights 128..255 (half 1)              */
/*     [8,136) 128 bytes of nibbles; weight j of the block sits in payload   */
/*             byte j/2, low nibble for even j                               */
/*   w_j = q_j * scale[h] + zero[h], q_j in 0..15,                           */
/*   h = 1 when the weight's payload byte offset is >= 64 (j >= 128).        */
/*   Row o holds I/256 blocks back to back; I must be a multiple of 256.     */
/* ------------------------------------------------------------------------ */

static uint32_t le32(const uint8_t *p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

double oracle_mq4v2_weight(const uint8_t *block, int j)
{
    int byte_off = j / 2;                    /* offset within the payload */
    int h = byte_off >= 64 ? 1 : 0;
    uint32_t hd = le32(block + 4 * h);
    double sc = oracle_f16_value((uint16_t)(hd & 0xFFFFu));
    double z = oracle_f16_value((uint16_t)(hd >> 16));
    uint8_t byte = block[8 + byte_off];
    int q = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return (double)q * sc + z;
}

void oracle_qgemv_mq4v2(double *y, double *mag, const uint16_t *x, const uint8_t *blocks,
                        int S, int I, int O)
{
    size_t nb = (size_t)I / 256;
    for (int s = 0; s < S; ++s) {
        for (int o = 0; o < O; ++o) {
            double acc = 0.0, m = 0.0;
            for (size_t b = 0; b < nb; ++b) {
                const uint8_t *blk = blocks + ((size_t)o * nb + b) * 136;
                for (int j = 0; j < 256; ++j) {
                    double t = oracle_mq4v2_weight(blk, j) *
                               oracle_bf16_value(x[(size_t)s * I + b * 256 + (size_t)j]);
                    acc += t;
                    m += fabs(t);
                }
            }
            y[(size_t)s * O + o] = acc;
            mag[(size_t)s * O + o] = m;
        }
    }
}

/* Encoder ([hipfire MQ4V2] section 3).  Per 128-weight half:
 *   lo = min, hi = max, step = (hi - lo) / 15       (binary32)
 *   scale = f16(step), zero = f16(lo)               (stored)
 *   st = f32(scale), z = f32(zero)                  (round-tripped)
 *   q = clamp(rint((w - z) / st), 0, 15)            (binary32)
 * A constant half (hi == lo) stores scale 0, zero f16(lo) and q = 0.
 * Reading taken where the page is silent: a half whose rounded step is 0
 * (step below half the smallest fp16 subnormal) is treated like a constant
 * half (q = 0) instead of dividing by zero.                                 */
void oracle_encode_mq4v2(uint8_t *blocks, const float *w, int O, int I)
{
    size_t nb = (size_t)I / 256;
    for (int o = 0; o < O; ++o) {
        for (size_t b = 0; b < nb; ++b) {
            uint8_t *blk = blocks + ((size_t)o * nb + b) * 136;
            const float *src = w + (size_t)o * I + b * 256;
            memset(blk, 0, 136);
            for (int h = 0; h < 2; ++h) {
                const float *hw = src + 128 * h;
                float lo = hw[0], hi = hw[0];
                for (int j = 1; j < 128; ++j) {
                    if (hw[j] < lo) lo = hw[j];
                    if (hw[j] > hi) hi = hw[j];
                }
                volatile float diff = hi - lo;
                volatile float step = diff / 15.0f;
                uint16_t sc16 = (hi == lo) ? (uint16_t)0 : oracle_f16_from_f32(step);
                uint16_t z16 = oracle_f16_from_f32(lo);
                float st = (float)oracle_f16_value(sc16);
                float z = (float)oracle_f16_value(z16);
                uint32_t hd = (uint32_t)sc16 | ((uint32_t)z16 << 16);
                blk[4 * h + 0] = (uint8_t)(hd & 0xFF);
                blk[4 * h + 1] = (uint8_t)((hd >> 8) & 0xFF);
                blk[4 * h + 2] = (uint8_t)((hd >> 16) & 0xFF);
                blk[4 * h + 3] = (uint8_t)((hd >> 24) & 0xFF);
                for (int j = 0; j < 128; ++j) {
                    int q = 0;
                    if (st != 0.0f) {
                        volatile float d = hw[j] - z;
                        volatile float r = d / st;
                        float qr = rintf(r);
                        if (qr < 0.0f) qr = 0.0f;
                        if (qr > 15.0f) qr = 15.0f;
                        q = (int)qr;
                    }
                    int jj = 128 * h + j;
                    uint8_t *byte = blk + 8 + jj / 2;
                    if (jj % 2 == 0)
                        *byte = (uint8_t)((*byte & 0xF0) | q);
                    else
                        *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MQ4 v1 (qt=13) and MQ4C pad (qt=45) ([hipfire MQ4V2] sections 1b, 1e)     */
/*   The same 136-byte block per 256 weights and the same nibble payload at  */
/*   [8,136) as MQ4-V2, with one header for all 256 weights of the block:    */
/*     v1:   [0,4) f32 scale, [4,8) f32 zero                                 */
/*     pad:  [0,2) fp16 scale, [2,4) fp16 zero, [4,8) zero bytes             */
/*   w_j = q_j * scale + zero.                                               */
/* ------------------------------------------------------------------------ */

/* Nibble of weight j of a 136-byte block: payload byte j/2 after the 8
 * header bytes, the low nibble for even j. */
static int mq4_payload_nibble(const uint8_t *block, int j)
{
    const uint8_t *payload = block + 8;
    uint8_t b = payload[j >> 1];
    return (j & 1) ? (b >> 4) : (b & 0xF);
}

static double f32_at(const uint8_t *p)
{
    uint32_t u = le32(p);
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_mq4v1_weight(const uint8_t *block, int j)
{
    double scale = f32_at(block);
    double zero = f32_at(block + 4);
    return (double)mq4_payload_nibble(block, j) * scale + zero;
}

double oracle_mq4c_weight(const uint8_t *block, int j)
{
    uint32_t pair = le32(block);
    double scale = oracle_f16_value((uint16_t)(pair & 0xFFFFu));
    double zero = oracle_f16_value((uint16_t)(pair >> 16));
    return (double)mq4_payload_nibble(block, j) * scale + zero;
}

/* y[s,o] = sum_j w(o, j) x[s, j] over the row's I/256 blocks, one block
 * after another; mag the same sum of |terms|. */
static void mq4_one_header_gemv(double (*weight)(const uint8_t *, int), double *y, double *mag,
                                const uint16_t *x, const uint8_t *blocks, int S, int I, int O)
{
    const size_t row_blocks = (size_t)I / 256;
    for (int s = 0; s < S; ++s)
        for (int o = 0; o < O; ++o) {
            double sum = 0.0, sum_abs = 0.0;
            const uint8_t *row = blocks + (size_t)o * row_blocks * 136;
            for (int i = 0; i < I; ++i) {
                double t = weight(row + (size_t)(i / 256) * 136, i % 256) *
                           oracle_bf16_value(x[(size_t)s * I + (size_t)i]);
                sum += t;
                sum_abs += fabs(t);
            }
            y[(size_t)s * O + o] = sum;
            mag[(size_t)s * O + o] = sum_abs;
        }
}

void oracle_qgemv_mq4v1(double *y, double *mag, const uint16_t *x, const uint8_t *blocks, int S, int I,
                        int O)
{
    mq4_one_header_gemv(oracle_mq4v1_weight, y, mag, x, blocks, S, I, O);
}

void oracle_qgemv_mq4c(double *y, double *mag, const uint16_t *x, const uint8_t *blocks, int S, int I,
                       int O)
{
    mq4_one_header_gemv(oracle_mq4c_weight, y, mag, x, blocks, S, I, O);
}

/* Encoders: the MQ4 rule ("level placement uniform over [min, max]",
 * [hipfire MQ4V2] section 1c) over the whole 256-weight block.
 *   lo = min, hi = max, step = (hi - lo) / 15         (binary32)
 *   v1:  scale = step, zero = lo stored as f32; q against them
 *   pad: scale = f16(step), zero = f16(lo) stored; q against the
 *        round-tripped values; bytes [4,8) zero
 *   q = clamp(rint((w - zero) / scale), 0, 15)        (binary32)
 * A constant block (hi == lo), or one whose stored step is 0, stores
 * scale 0 and q = 0 (the MQ4-V2 encoder's reading).                       */
static void mq4_encode_one_header(uint8_t *blocks, const float *w, int O, int I, int fp16_header)
{
    const size_t row_blocks = (size_t)I / 256;
    for (int o = 0; o < O; ++o)
        for (size_t b = 0; b < row_blocks; ++b) {
            uint8_t *out = blocks + ((size_t)o * row_blocks + b) * 136;
            const float *v = w + (size_t)o * I + b * 256;
            float lo = v[0], hi = v[0];
            for (int j = 1; j < 256; ++j) {
                lo = v[j] < lo ? v[j] : lo;
                hi = v[j] > hi ? v[j] : hi;
            }
            volatile float span = hi - lo;
            volatile float step = span / 15.0f;
            float scale, zero;
            uint32_t word0, word1;
            if (fp16_header) {
                uint16_t s16 = (hi == lo) ? (uint16_t)0 : oracle_f16_from_f32(step);
                uint16_t z16 = oracle_f16_from_f32(lo);
                scale = (float)oracle_f16_value(s16);
                zero = (float)oracle_f16_value(z16);
                word0 = (uint32_t)s16 | ((uint32_t)z16 << 16);
                word1 = 0u;
            } else {
                scale = (hi == lo) ? 0.0f : step;
                zero = lo;
                memcpy(&word0, &scale, 4);
                memcpy(&word1, &zero, 4);
            }
            for (int k = 0; k < 4; ++k) {
                out[k] = (uint8_t)(word0 >> (8 * k));
                out[4 + k] = (uint8_t)(word1 >> (8 * k));
            }
            for (int j = 0; j < 256; j += 2) {
                int q2[2];
                for (int e = 0; e < 2; ++e) {
                    int q = 0;
                    if (scale != 0.0f) {
                        volatile float d = v[j + e] - zero;
                        volatile float r = d / scale;
                        float qf = rintf(r);
                        q = qf < 0.0f ? 0 : qf > 15.0f ? 15 : (int)qf;
                    }
                    q2[e] = q;
                }
                out[8 + j / 2] = (uint8_t)(q2[0] | (q2[1] << 4));
            }
        }
}

void oracle_encode_mq4v1(uint8_t *blocks, const float *w, int O, int I)
{
    mq4_encode_one_header(blocks, w, O, I, 0);
}

void oracle_encode_mq4c(uint8_t *blocks, const float *w, int O, int I)
{
    mq4_encode_one_header(blocks, w, O, I, 1);
}

/* ------------------------------------------------------------------------ */
/* Routed experts ([colibri #457] section 7: the batched routed-expert path  */
/* walks a per-expert pointer array with one format and group size per       */
/* tensor; [hipfire MQ4V2] section 9: MoE decode on MQ4-V2).                 */
/*   Slot r multiplies the expert ids[r] of the table with its own           */
/*   activations x_r = x + r * x_slot_stride (elements; 0: every slot reads  */
/*   the same x) into y_r = y + r * S * O:  y_r = W_{ids[r]} x_r, the         */
/*   single-matrix definition of `fmt` applied slot by slot.  A slot whose   */
/*   id names no expert of the table has no value: NaN.                      */
/* ------------------------------------------------------------------------ */
void oracle_qgemv_moe(int fmt, double *y, double *mag, const void *x, size_t x_slot_stride,
                      const void *const *w, const float *const *scales, int n_experts,
                      const int *ids, int n_slots, int S, int I, int O, int gs)
{
    const size_t out_n = (size_t)S * O;
    for (int r = 0; r < n_slots; ++r) {
        double *yr = y + (size_t)r * out_n;
        double *mr = mag + (size_t)r * out_n;
        const int id = ids[r];
        const size_t xo = (size_t)r * x_slot_stride;
        const uint8_t *we = (id >= 0 && id < n_experts) ? (const uint8_t *)w[id] : NULL;
        if (we == NULL) {
            for (size_t k = 0; k < out_n; ++k)
                yr[k] = mr[k] = NAN;
            continue;
        }
        switch (fmt) {
        case 4:
            oracle_qgemv_i4g(yr, mr, (const float *)x + xo, we, scales[id], S, I, O, gs);
            break;
        case 7:
            oracle_qgemv_fp8b128(yr, mr, (const uint16_t *)x + xo, we, scales[id], S, I, O);
            break;
        case 71: /* fmt=7 with UE8M0 scales: the table's scale pointer holds the bytes */
            oracle_qgemv_fp8ue8m0(yr, mr, (const uint16_t *)x + xo, we, (const uint8_t *)scales[id], S, I, O);
            break;
        case 13:
            oracle_qgemv_mq4v1(yr, mr, (const uint16_t *)x + xo, we, S, I, O);
            break;
        case 44:
            oracle_qgemv_mq4v2(yr, mr, (const uint16_t *)x + xo, we, S, I, O);
            break;
        case 45:
            oracle_qgemv_mq4c(yr, mr, (const uint16_t *)x + xo, we, S, I, O);
            break;
        default:
            for (size_t k = 0; k < out_n; ++k)
                yr[k] = mr[k] = NAN;
        }
    }
}

/* Routed-expert prefill: tokens sorted by expert; group g multiplies the rows
 * [off[g], off[g+1]) of X (bf16 [M, I]) by the expert group_expert[g] into the
 * same rows of Y, with the single-matrix prefill definition of `fmt` (the
 * fmt=4 GEMM; the GEMV definitions of the other formats with S = the group's
 * rows).  Rows that no group covers are left untouched.                     */
void oracle_qgemm_moe(int fmt, double *Y, double *mag, const uint16_t *X, const void *const *w,
                      const float *const *scales, int n_experts, const int *group_expert,
                      const int *off, int n_groups, int I, int O, int gs)
{
    for (int g = 0; g < n_groups; ++g) {
        const int e = group_expert[g];
        const int m = off[g + 1] - off[g];
        if (m <= 0 || e < 0 || e >= n_experts)
            continue;
        double *yg = Y + (size_t)off[g] * O;
        double *mg = mag + (size_t)off[g] * O;
        const uint16_t *xg = X + (size_t)off[g] * I;
        const uint8_t *we = (const uint8_t *)w[e];
        switch (fmt) {
        case 4:
            oracle_qgemm_i4g(yg, mg, xg, we, scales[e], m, I, O, gs);
            break;
        case 7:
            oracle_qgemv_fp8b128(yg, mg, xg, we, scales[e], m, I, O);
            break;
        case 71:
            oracle_qgemv_fp8ue8m0(yg, mg, xg, we, (const uint8_t *)scales[e], m, I, O);
            break;
        case 13:
            oracle_qgemv_mq4v1(yg, mg, xg, we, m, I, O);
            break;
        case 44:
            oracle_qgemv_mq4v2(yg, mg, xg, we, m, I, O);
            break;
        case 45:
            oracle_qgemv_mq4c(yg, mg, xg, we, m, I, O);
            break;
        default:
            break;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Seeded sign-FWHT over 256-element blocks ([hipfire MQ4V2] sections 1, 1d, */
/* 3: the MQ line rotates every 256-block with a signed Walsh-Hadamard       */
/* transform before quantizing; the rotated activation is consumed by the    */
/* GEMV).  Reading: v <- H_256 (d . v) / 16 with H_256 the Sylvester         */
/* Hadamard matrix in natural order and d in {+1,-1}^256 a sign vector       */
/* passed in by the caller.  H/16 is orthonormal, so applying the transform  */
/* to both a weight row and the activation preserves every dot product.     */
/* The butterfly is the fast Walsh-Hadamard algorithm itself, in double.     */
/* ------------------------------------------------------------------------ */
void oracle_fwht256(float *out, const float *in, const int8_t *signs, size_t nblocks)
{
    double v[256];
    for (size_t b = 0; b < nblocks; ++b) {
        for (int j = 0; j < 256; ++j)
            v[j] = (double)signs[j] * (double)in[b * 256 + (size_t)j];
        for (int len = 1; len < 256; len <<= 1) {
            for (int base = 0; base < 256; base += 2 * len) {
                for (int j = base; j < base + len; ++j) {
                    double a = v[j], c = v[j + len];
                    v[j] = a + c;
                    v[j + len] = a - c;
                }
            }
        }
        for (int j = 0; j < 256; ++j)
            out[b * 256 + (size_t)j] = (float)(v[j] / 16.0);
    }
}

/* Inverse of oracle_fwht256: H/16 is symmetric and orthonormal, so the
 * inverse applies the same transform and then the same signs again.         */
void oracle_ifwht256(float *out, const float *in, const int8_t *signs, size_t nblocks)
{
    double v[256];
    for (size_t b = 0; b < nblocks; ++b) {
        for (int j = 0; j < 256; ++j)
            v[j] = (double)in[b * 256 + (size_t)j];
        for (int len = 1; len < 256; len <<= 1) {
            for (int base = 0; base < 256; base += 2 * len) {
                for (int j = base; j < base + len; ++j) {
                    double a = v[j], c = v[j + len];
                    v[j] = a + c;
                    v[j + len] = a - c;
                }
            }
        }
        for (int j = 0; j < 256; ++j)
            out[b * 256 + (size_t)j] = (float)((double)signs[j] * v[j] / 16.0);
    }
}
