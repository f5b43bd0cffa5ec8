/* synth.c -- host implementation of the seeded input generators (synth.h). */
#include "synth.h"

#include <stdlib.h>
#include <string.h>

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t draw(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * SYNTH_GAMMA); }

void synth_xorshift_f32(uint64_t *state, int64_t count, float *out)
{
    uint64_t s = *state;
    for (int64_t j = 0; j < count; ++j) {
        s ^= s << 13;
        s ^= s >> 7;
        s ^= s << 17;
        float r = (float)(s >> 11) / (float)(1ULL << 53) * 2.0f - 1.0f;
        out[j] = r;
    }
    *state = s;
}

static float uniform_at(uint64_t seed, uint64_t i)
{
    int32_t u = (int32_t)(draw(seed, i) >> 40);
    int32_t v = 2 * u + 1 - (1 << 24);
    return (float)v * 0x1p-24f;
}

static float normal_at(uint64_t seed, uint64_t i)
{
    int64_t sum = 0;
    for (int j = 0; j < 6; ++j) {
        uint64_t d = draw(seed, 6 * i + (uint64_t)j);
        sum += (int64_t)(d >> 40);
        sum += (int64_t)((d >> 16) & 0xFFFFFFULL);
    }
    int32_t v = (int32_t)(sum - 6LL * (1LL << 24));
    return (float)v * 0x1p-24f;
}

void synth_uniform_f32(uint64_t seed, int64_t start, int64_t count, float scale, float *out)
{
    for (int64_t j = 0; j < count; ++j) out[j] = scale * uniform_at(seed, (uint64_t)(start + j));
}

void synth_normal_f32(uint64_t seed, int64_t start, int64_t count, float sigma, float *out)
{
    for (int64_t j = 0; j < count; ++j) out[j] = sigma * normal_at(seed, (uint64_t)(start + j));
}

void synth_normal_rows_f32(uint64_t seed, int64_t C, int64_t r0, int64_t r1, float sigma,
                           const int32_t *cols, int64_t ncols, float factor, float *out)
{
    for (int64_t r = r0; r < r1; ++r) {
        float *row = out + (r - r0) * C;
        synth_normal_f32(seed, r * C, C, sigma, row);
        for (int64_t j = 0; j < ncols; ++j) row[cols[j]] = row[cols[j]] * factor;
    }
}

void synth_f32_to_bf16(const float *in, int64_t count, uint16_t *out)
{
    for (int64_t j = 0; j < count; ++j) {
        uint32_t b;
        memcpy(&b, &in[j], 4);
        if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) {
            out[j] = (uint16_t)((b >> 16) | 0x0040u); /* quiet NaN */
            continue;
        }
        b += 0x7FFFu + ((b >> 16) & 1u);
        out[j] = (uint16_t)(b >> 16);
    }
}

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

void synth_sample_without_replacement(uint64_t seed, int64_t n, int64_t count, int32_t *out)
{
    int32_t *perm = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    for (int64_t i = 0; i < n; ++i) perm[i] = (int32_t)i;
    for (int64_t i = 0; i < count; ++i) {
        uint64_t r = draw(seed, (uint64_t)i) % (uint64_t)(n - i);
        int64_t j = i + (int64_t)r;
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    memcpy(out, perm, (size_t)count * sizeof(int32_t));
    free(perm);
    qsort(out, (size_t)count, sizeof(int32_t), cmp_i32);
}
