/*
 * oq4.c -- CPU oracle (test infrastructure only; see oq4.h).
 *
 * Follows the page "Weight quantization", sections "How it works" and "Code".
 * Build with contraction off so every f32 expression rounds exactly where the
 * page's f32 code rounds:   gcc -O2 -std=c99 -ffp-contract=off -fPIC -shared
 *
 * OQ4_MUTANT (compile-time, default 0) plants one known mistake so that the
 * test suite can show its pins catch it.  It is never set in a normal build.
 */
#include "oq4.h"

#include <float.h>
#include <math.h>
#include <stddef.h>
#include <string.h>

#ifndef OQ4_MUTANT
#define OQ4_MUTANT 0
#endif

int oq4_mutant(void) { return OQ4_MUTANT; }

/* Rust's f32::clamp(lo, hi): below lo -> lo, above hi -> hi, else unchanged. */
static float clampf(float v, float lo, float hi)
{
    if (v < lo) return lo;
    if (v > hi) return hi;
    return v;
}

/* "round" on the page is Rust's f32::round: ties go away from zero, which is
 * C99 roundf.  (Mutants 1/2 swap in ties-to-even, the torch/Python rule.) */
static float round_code(float v)
{
#if OQ4_MUTANT == 1
    return rintf(v);
#else
    return roundf(v);
#endif
}

static float round_zero(float v)
{
#if OQ4_MUTANT == 2
    return rintf(v);
#else
    return roundf(v);
#endif
}

/* Where code `v` of flat weight index `idx` goes: byte idx/2, low nibble for
 * an even index ("low nibble = even index" in the page's quantize). */
static void put_code(uint8_t *packed, int64_t idx, uint8_t v)
{
#if OQ4_MUTANT == 3
    packed[idx / 2] |= (uint8_t)(v << ((1 - (idx & 1)) * 4));
#else
    packed[idx / 2] |= (uint8_t)(v << ((idx & 1) * 4));
#endif
}

static uint8_t get_code(const uint8_t *packed, int64_t idx)
{
    /* the inverse of put_code for the real layout */
    uint8_t b = packed[idx / 2];
    return (idx & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0x0F);
}

int oq4_quantize_g(const float *w, int64_t N, int64_t K, int64_t G,
                   uint8_t *packed, float *scale, uint8_t *zero)
{
    if (G <= 0 || K % G != 0 || ((N * K) & 1)) return -1;
    memset(packed, 0, (size_t)(N * K / 2));

    /* The page walks the flat weight vector in chunks of G; with K % G == 0 a
     * chunk never straddles two rows, so chunk gi = n*(K/G) + g. */
    const int64_t ngroups = N * K / G;
    for (int64_t gi = 0; gi < ngroups; ++gi) {
        const float *grp = w + gi * G;

        /* 1. group minimum and maximum, folded from (f32::MAX, f32::MIN) */
        float lo = FLT_MAX, hi = -FLT_MAX;
        for (int64_t j = 0; j < G; ++j) {
            lo = fminf(lo, grp[j]);
            hi = fmaxf(hi, grp[j]);
        }
        /* 2. widen the range to contain 0 so that 0 is exactly representable */
#if OQ4_MUTANT != 4
        lo = fminf(lo, 0.0f);
        hi = fmaxf(hi, 0.0f);
#endif
        /* 3. scale = (max - min) / (2^b - 1), or 1 when the range is empty */
#if OQ4_MUTANT == 5
        float s = (hi > lo) ? (hi - lo) / 16.0f : 1.0f;
#else
        float s = (hi > lo) ? (hi - lo) / 15.0f : 1.0f;
#endif
        /* 4. zero = round(-min / scale), clamped to [0, 15] */
#if OQ4_MUTANT == 7
        float z = clampf(round_zero(lo / s), 0.0f, 15.0f);
#else
        float z = clampf(round_zero(-lo / s), 0.0f, 15.0f);
#endif
        scale[gi] = s;
        zero[gi] = (uint8_t)z;

        /* 5. q = clamp(round(w / scale) + zero, 0, 15), then pack */
        for (int64_t j = 0; j < G; ++j) {
#if OQ4_MUTANT == 6
            float qf = clampf(round_code(grp[j] / s + z), 0.0f, 15.0f);
#else
            float qf = clampf(round_code(grp[j] / s) + z, 0.0f, 15.0f);
#endif
            put_code(packed, gi * G + j, (uint8_t)qf);
        }
    }
    return 0;
}

int oq4_quantize(const float *w, int64_t N, int64_t K,
                 uint8_t *packed, float *scale, uint8_t *zero)
{
    return oq4_quantize_g(w, N, K, OQ4_G, packed, scale, zero);
}

/* Symmetric variant (page "Quantization", hritesh-sonawane.github.io notes,
 * section "How it really works", "The mechanics: scale, round, clamp", and
 * its "Code" section, function int_quant; page "LLM Quantization Architecture
 * in Depth", the group-wise symmetric listing):
 *   s = max|w| / 7, or 1 when that is 0     (the "or 1.0" of int_quant)
 *   q = clamp(round(w / s), -8, 7)          (round = ties to even, as both
 *                                            pages' round() does)
 *   w_hat = q * s
 * Stored in the same containers as the asymmetric scheme: code q + 8 in the
 * nibble and zero = 8, so that (code - zero) * s == q * s exactly. */
static float round_sym(float v)
{
#if OQ4_MUTANT == 12
    return roundf(v);
#else
    return rintf(v);
#endif
}

int oq4_quantize_sym_g(const float *w, int64_t N, int64_t K, int64_t G,
                       uint8_t *packed, float *scale, uint8_t *zero)
{
    if (G <= 0 || K % G != 0 || ((N * K) & 1)) return -1;
    memset(packed, 0, (size_t)(N * K / 2));
    const int64_t ngroups = N * K / G;
    for (int64_t gi = 0; gi < ngroups; ++gi) {
        const float *grp = w + gi * G;
        /* 1. largest magnitude of the group */
        float amax = 0.0f;
        for (int64_t j = 0; j < G; ++j) amax = fmaxf(amax, fabsf(grp[j]));
        /* 2. scale = max|w| / (2^(b-1) - 1), 1 when the quotient is 0 */
#if OQ4_MUTANT == 13
        float s = amax / 8.0f;
#else
        float s = amax / 7.0f;
#endif
        if (s == 0.0f) s = 1.0f;
        scale[gi] = s;
#if OQ4_MUTANT == 14
        const float off = 7.0f;
#else
        const float off = 8.0f;
#endif
        zero[gi] = 8;
        /* 3. q = clamp(round(w / s), -8, 7), stored as q + 8 */
        for (int64_t j = 0; j < G; ++j) {
            float qf = clampf(round_sym(grp[j] / s), -8.0f, 7.0f);
            put_code(packed, gi * G + j, (uint8_t)(qf + off));
        }
    }
    return 0;
}

int oq4_quantize_sym(const float *w, int64_t N, int64_t K,
                     uint8_t *packed, float *scale, uint8_t *zero)
{
    return oq4_quantize_sym_g(w, N, K, OQ4_G, packed, scale, zero);
}

/* w_hat = (q - zero) * scale  ("How it works", last formula).  Both factors
 * are exact in double, and so is their product (4-bit x 24-bit). */
static double what_at(const uint8_t *packed, const float *scale, const uint8_t *zero,
                      int64_t K, int64_t G, int64_t n, int64_t k)
{
    int64_t gi = n * (K / G) + k / G;
#if OQ4_MUTANT == 11
    gi = n * (K / G) + ((k + G / 2) / G) % (K / G);
#endif
    double q = (double)get_code(packed, n * K + k);
    double z = (double)zero[gi];
#if OQ4_MUTANT == 9
    return (q + z) * (double)scale[gi];
#else
    return (q - z) * (double)scale[gi];
#endif
}

void oq4_dequant_g(const uint8_t *packed, const float *scale, const uint8_t *zero,
                   int64_t N, int64_t K, int64_t G, double *w_hat)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w_hat[n * K + k] = what_at(packed, scale, zero, K, G, n, k);
}

void oq4_dot_naive(const float *x, int64_t M,
                   const uint8_t *packed, const float *scale, const uint8_t *zero,
                   int64_t N, int64_t K, int64_t n0, int64_t n1,
                   double *y, double *absdot)
{
    const int64_t R = n1 - n0;
    (void)N;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = n0; n < n1; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
#if OQ4_MUTANT == 10
                /* transposed operand: reads w_hat[k][n] (square matrices) */
                double wh = what_at(packed, scale, zero, K, OQ4_G, k % N, n % K);
#else
                double wh = what_at(packed, scale, zero, K, OQ4_G, n, k);
#endif
                double p = wh * (double)x[m * K + k];
                acc += p;
                aacc += fabs(p);
            }
            y[m * R + (n - n0)] = acc;
            if (absdot) absdot[m * R + (n - n0)] = aacc;
        }
    }
}

void oq4_dot_factored(const float *x, int64_t M,
                      const uint8_t *packed, const float *scale, const uint8_t *zero,
                      int64_t N, int64_t K, int64_t n0, int64_t n1, float *y)
{
    const int64_t R = n1 - n0, NG = K / OQ4_G;
    (void)N;
    for (int64_t m = 0; m < M; ++m) {
        const float *xr = x + m * K;
        for (int64_t n = n0; n < n1; ++n) {
            float acc = 0.0f;
            for (int64_t g = 0; g < NG; ++g) {
                const int64_t gi = n * NG + g;
                const uint8_t *bytes = packed + (n * K + g * OQ4_G) / 2;
                const float *xg = xr + g * OQ4_G;
                float qx = 0.0f, sx = 0.0f;
                for (int64_t b = 0; b < OQ4_G / 2; ++b) {
                    float x0 = xg[2 * b], x1 = xg[2 * b + 1];
                    qx += (float)(bytes[b] & 0x0F) * x0 + (float)(bytes[b] >> 4) * x1;
                    sx += x0 + x1;
                }
#if OQ4_MUTANT == 8
                acc += scale[gi] * qx;
#else
                acc += scale[gi] * (qx - (float)zero[gi] * sx);
#endif
            }
            y[m * R + (n - n0)] = acc;
        }
    }
}

void oq4_xsum(const float *x, int64_t M, int64_t K, double *xsum)
{
    const int64_t NG = K / OQ4_G;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t g = 0; g < NG; ++g) {
            double s = 0.0;
            for (int64_t j = 0; j < OQ4_G; ++j) s += (double)x[m * K + g * OQ4_G + j];
            xsum[m * NG + g] = s;
        }
}

/* ---------------------------------------------------------------------------
 * Compact metadata (page "Weight quantization", section "Code": the bits per
 * weight it prints count each scale as 16 bits and each zero as 4 bits;
 * section "Complexity and constants": int4 g128 with an fp16 scale and a
 * 4-bit zero; "Implementation notes": keep scales in fp16/bf16).  The codes
 * and zeros are the canonical ones; the scale is stored rounded once to IEEE
 * binary16 (round to nearest, ties to even), and the zeros two per byte. */

/* f32 -> binary16 bits, round to nearest even; overflow gives infinity. */
uint16_t oq4_f16_bits(float v)
{
    uint32_t x;
    memcpy(&x, &v, sizeof x);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const uint32_t ex = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;
    if (ex == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
    const int e = (int)ex - 127 + 15;  /* binary16 biased exponent */
    if (e >= 31) return (uint16_t)(sign | 0x7C00u);
    if (e <= 0) {
        /* binary16 subnormal (or zero): units of 2^-24 */
        if (ex == 0) return (uint16_t)sign;  /* f32 subnormals are below 2^-126 */
        man |= 0x800000u;
        const int shift = 14 - e;
        if (shift > 24) return (uint16_t)sign;
        uint32_t q = man >> shift;
        const uint32_t rem = man & ((1u << shift) - 1u), half = 1u << (shift - 1);
#if OQ4_MUTANT != 15
        if (rem > half || (rem == half && (q & 1u))) ++q;
#endif
        return (uint16_t)(sign | q);
    }
    uint32_t q = ((uint32_t)e << 10) | (man >> 13);
    const uint32_t rem = man & 0x1FFFu;
#if OQ4_MUTANT != 15
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) ++q;  /* a carry may reach infinity */
#endif
    return (uint16_t)(sign | q);
}

/* binary16 bits -> f32 (exact). */
float oq4_f16_value(uint16_t h)
{
    const int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(sign ? -v : v);
}

void oq4_compact_meta(const float *scale, const uint8_t *zero, int64_t N, int64_t NG,
                      uint16_t *scale16, uint8_t *zero4)
{
    const int64_t ZB = (NG + 1) / 2;
    memset(zero4, 0, (size_t)(N * ZB));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < NG; ++g) {
            scale16[n * NG + g] = oq4_f16_bits(scale[n * NG + g]);
#if OQ4_MUTANT == 16
            const int hi = !(g & 1);
#else
            const int hi = (int)(g & 1);
#endif
            zero4[n * ZB + g / 2] |= (uint8_t)((zero[n * NG + g] & 0x0F) << (4 * hi));
        }
}

void oq4_expand_meta(const uint16_t *scale16, const uint8_t *zero4, int64_t N, int64_t NG,
                     float *scale, uint8_t *zero)
{
    const int64_t ZB = (NG + 1) / 2;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < NG; ++g) {
            scale[n * NG + g] = oq4_f16_value(scale16[n * NG + g]);
            const uint8_t b = zero4[n * ZB + g / 2];
            zero[n * NG + g] = (g & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0x0F);
        }
}

