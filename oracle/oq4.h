/*
 * oq4.h -- CPU oracle for group-wise INT4 weight quantization (asymmetric,
 * and the symmetric variant) and the weight-only (W4A16) matrix-vector
 * product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or execute this code: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no source, header, table or
 * helper with the CUDA library and does not know the library's kernel layout.
 *
 * Source of every definition: the web page "Weight quantization"
 * (tirogla.com, ml-training/weight-quantization), section "How it works"
 * (the four formulas for scale, zero, q and w_hat, and the factored group dot
 * product) and section "Code" (functions `quantize` and `dot`, struct `Q4`).
 *
 * Storage contract (the page's struct Q4):
 *   w       f32 [N][K], row-major, groups of G=128 consecutive weights along K
 *   packed  u8  [N*K/2]   two codes per byte; the even flat index n*K+k sits
 *                         in the LOW nibble, the odd one in the high nibble
 *   scale   f32 [N][K/G]  one scale per group
 *   zero    u8  [N][K/G]  one zero point per group, 0..15
 *
 * Parity status of each function (what pins it) is listed in the test suite's
 * oracle pin tests; every function below is pinned.
 */
#ifndef OQ4_H
#define OQ4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OQ4_G 128

/* Round-to-nearest asymmetric quantization with group size G (the page fixes
 * G=128; smaller G is used only by brute-force tests on tiny groups).
 * Returns 0, or -1 if K % G != 0 or N*K is odd. packed is zero-filled here. */
int oq4_quantize_g(const float *w, int64_t N, int64_t K, int64_t G,
                   uint8_t *packed, float *scale, uint8_t *zero);

/* Same with G = 128. */
int oq4_quantize(const float *w, int64_t N, int64_t K,
                 uint8_t *packed, float *scale, uint8_t *zero);

/* Symmetric round-to-nearest with group size G: s = max|w|/7 (1 when that
 * quotient is 0), q = clamp(rint(w/s), -8, 7) with ties to even, stored as
 * code q + 8 with zero = 8 in the same containers, so the dequantization and
 * products below serve both schemes.  Source: page "Quantization"
 * (hritesh-sonawane.github.io notes), "How it really works" and "Code"
 * (int_quant); page "LLM Quantization Architecture in Depth", the group-wise
 * symmetric listing.  Returns 0, or -1 on a bad shape (as above). */
int oq4_quantize_sym_g(const float *w, int64_t N, int64_t K, int64_t G,
                       uint8_t *packed, float *scale, uint8_t *zero);
int oq4_quantize_sym(const float *w, int64_t N, int64_t K,
                     uint8_t *packed, float *scale, uint8_t *zero);

/* w_hat[n][k] = (q - zero) * scale, exactly, in double. */
void oq4_dequant_g(const uint8_t *packed, const float *scale, const uint8_t *zero,
                   int64_t N, int64_t K, int64_t G, double *w_hat);

/* Plain definition of the product for output rows n in [n0, n1):
 *   y[m][n-n0]      = sum_k w_hat[n][k] * x[m][k]      (double)
 *   absdot[m][n-n0] = sum_k |w_hat[n][k] * x[m][k]|    (double, for tolerances)
 * x is f32 [M][K]; bf16/fp16 activations are widened exactly by the caller.
 * absdot may be NULL. */
void oq4_dot_naive(const float *x, int64_t M,
                   const uint8_t *packed, const float *scale, const uint8_t *zero,
                   int64_t N, int64_t K, int64_t n0, int64_t n1,
                   double *y, double *absdot);

/* The page's factored dot product, in f32 as the page writes it, per group:
 *   qx += q_even*x_even + q_odd*x_odd;  sx += x_even + x_odd;
 *   acc += scale * (qx - zero*sx)
 * generalised to M activation rows and output rows [n0, n1). y is f32. */
void oq4_dot_factored(const float *x, int64_t M,
                      const uint8_t *packed, const float *scale, const uint8_t *zero,
                      int64_t N, int64_t K, int64_t n0, int64_t n1, float *y);

/* Activation group sums: xsum[m][g] = sum_{k in group g} x[m][k] (double). */
void oq4_xsum(const float *x, int64_t M, int64_t K, double *xsum);

/* Compact metadata (page "Weight quantization": the bits-per-weight formula
 * of section "Code" counts 16-bit scales and 4-bit zeros; "Complexity and
 * constants": fp16 scale + 4-bit zero; "Implementation notes": scales in
 * fp16/bf16).  Same codes and zeros as the canonical form; each scale
 * stored as binary16, rounded once to nearest even; zeros two per byte
 * (low nibble = even group).  scale16 [N][NG], zero4 [N][ceil(NG/2)].  The
 * products of a compact weight are those of the canonical containers that
 * oq4_expand_meta returns (the binary16 scale widened exactly). */
uint16_t oq4_f16_bits(float v);
float oq4_f16_value(uint16_t h);
void oq4_compact_meta(const float *scale, const uint8_t *zero, int64_t N, int64_t NG,
                      uint16_t *scale16, uint8_t *zero4);
void oq4_expand_meta(const uint16_t *scale16, const uint8_t *zero4, int64_t N, int64_t NG,
                     float *scale, uint8_t *zero);

/* Mutation id this build was compiled with (0 = the real oracle). */
int oq4_mutant(void);

#ifdef __cplusplus
}
#endif
#endif
