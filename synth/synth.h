/*
 * synth.h -- seeded synthetic-input generators shared by the oracle side and
 * the GPU side of the tests and the benchmark.  Holds none of the
 * quantization or matmul arithmetic: only random numbers and dtype rounding.
 *
 * Two generators:
 *  - the page's xorshift64 stream (shifts 13, 7, 17; seed 0x9E3779B97F4A7C15;
 *    value (state >> 11) as f32 / 2^53 as f32 * 2 - 1), page "Weight
 *    quantization", section "Code", function `main`.  Sequential, host only.
 *  - a counter-based generator: output i of SplitMix64 (Steele, Lea, Flood,
 *    "Fast splittable pseudorandom number generators", OOPSLA 2014; the
 *    public-domain splitmix64.c of S. Vigna) started at state `seed`, i.e.
 *    mix64(seed + (i + 1) * 0x9E3779B97F4A7C15).  Implemented identically
 *    here (host C) and in synth_dev.cu (CUDA), bit for bit.
 *
 * Derived draws (all integer arithmetic until one exact or RNE conversion):
 *  - uniform(i) in (-1, 1):  u = top 24 bits of draw i;
 *                            (float)(2u + 1 - 2^24) * 2^-24        (exact)
 *  - normal(i) ~ N(0, 1):    Irwin-Hall sum of 12 24-bit integers taken from
 *                            draws 6i..6i+5 (bits 63..40 and 39..16 of each),
 *                            minus 6*2^24, converted once to f32 (RNE),
 *                            times 2^-24; support is +-6.
 */
#ifndef Q4SYNTH_H
#define Q4SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL
#define SYNTH_PAGE_SEED 0x9E3779B97F4A7C15ULL

/* The page's xorshift stream: writes `count` draws in [-1, 1) and advances
 * *state. */
void synth_xorshift_f32(uint64_t *state, int64_t count, float *out);

/* out[j] = scale * uniform(start + j) */
void synth_uniform_f32(uint64_t seed, int64_t start, int64_t count, float scale, float *out);

/* out[j] = sigma * normal(start + j) */
void synth_normal_f32(uint64_t seed, int64_t start, int64_t count, float sigma, float *out);

/* Rows [r0, r1) of an R x C matrix whose element (r, c) is
 * sigma * normal(r*C + c), with columns listed in `cols` multiplied by
 * `factor` afterwards (f32 multiply). out is [r1-r0][C]. */
void synth_normal_rows_f32(uint64_t seed, int64_t C, int64_t r0, int64_t r1, float sigma,
                           const int32_t *cols, int64_t ncols, float factor, float *out);

/* Round-to-nearest-even f32 -> bf16 bit patterns. */
void synth_f32_to_bf16(const float *in, int64_t count, uint16_t *out);

/* `count` distinct values from [0, n) by a seeded partial Fisher-Yates
 * shuffle driven by the counter-based generator, returned in sorted order. */
void synth_sample_without_replacement(uint64_t seed, int64_t n, int64_t count, int32_t *out);

#ifdef __cplusplus
}
#endif
#endif
