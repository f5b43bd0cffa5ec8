/*
 * synth_dev.cu -- device implementation of the counter-based input generators
 * declared in synth.h (same definitions, bit for bit: integer arithmetic, one
 * RNE int->f32 conversion, exact power-of-two scaling, one f32 multiply).
 * Used to fill large synthetic weight and activation buffers directly in HBM.
 * Holds none of the quantization or matmul arithmetic.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t seed, uint64_t i)
{
    return mix64(seed + (i + 1) * SYNTH_GAMMA);
}

__device__ __forceinline__ float normal_at(uint64_t seed, uint64_t i)
{
    int64_t sum = 0;
#pragma unroll
    for (int j = 0; j < 6; ++j) {
        uint64_t d = draw(seed, 6 * i + (uint64_t)j);
        sum += (int64_t)(d >> 40);
        sum += (int64_t)((d >> 16) & 0xFFFFFFULL);
    }
    int32_t v = (int32_t)(sum - 6LL * (1LL << 24));
    return __fmul_rn(__int2float_rn(v), 0x1p-24f);
}

__device__ __forceinline__ float uniform_at(uint64_t seed, uint64_t i)
{
    int32_t u = (int32_t)(draw(seed, i) >> 40);
    int32_t v = 2 * u + 1 - (1 << 24);
    return __fmul_rn(__int2float_rn(v), 0x1p-24f);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f)
{
    uint32_t b = __float_as_uint(f);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

__global__ void k_normal_f32(float *out, int64_t count, uint64_t seed, int64_t start, float sigma,
                             const uint8_t *col_mask, int64_t C, float factor)
{
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < count;
         j += (int64_t)gridDim.x * blockDim.x) {
        float v = __fmul_rn(sigma, normal_at(seed, (uint64_t)(start + j)));
        if (col_mask && col_mask[(start + j) % C]) v = __fmul_rn(v, factor);
        out[j] = v;
    }
}

__global__ void k_uniform_f32(float *out, int64_t count, uint64_t seed, int64_t start, float scale)
{
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < count;
         j += (int64_t)gridDim.x * blockDim.x)
        out[j] = __fmul_rn(scale, uniform_at(seed, (uint64_t)(start + j)));
}

__global__ void k_normal_bf16(uint16_t *out, int64_t count, uint64_t seed, int64_t start, float sigma)
{
    for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < count;
         j += (int64_t)gridDim.x * blockDim.x)
        out[j] = f32_to_bf16_rne(__fmul_rn(sigma, normal_at(seed, (uint64_t)(start + j))));
}

static int grid_for(int64_t count)
{
    int64_t b = (count + 255) / 256;
    return (int)(b < 152 * 64 ? (b < 1 ? 1 : b) : 152 * 64);
}

extern "C" {

/* out[j] = sigma * normal(start + j), j < count; when col_mask (device, C
 * bytes) is given, elements whose column (start + j) % C is flagged are then
 * multiplied by factor.  Returns a cudaError_t value. */
int synth_dev_normal_f32(float *out, int64_t count, uint64_t seed, int64_t start, float sigma,
                         const uint8_t *col_mask, int64_t C, float factor, cudaStream_t s)
{
    if (count <= 0) return 0;
    k_normal_f32<<<grid_for(count), 256, 0, s>>>(out, count, seed, start, sigma, col_mask,
                                                 C > 0 ? C : 1, factor);
    return (int)cudaGetLastError();
}

int synth_dev_uniform_f32(float *out, int64_t count, uint64_t seed, int64_t start, float scale,
                          cudaStream_t s)
{
    if (count <= 0) return 0;
    k_uniform_f32<<<grid_for(count), 256, 0, s>>>(out, count, seed, start, scale);
    return (int)cudaGetLastError();
}

/* out[j] = bf16_rne(sigma * normal(start + j)) as raw bf16 bits. */
int synth_dev_normal_bf16(uint16_t *out, int64_t count, uint64_t seed, int64_t start, float sigma,
                          cudaStream_t s)
{
    if (count <= 0) return 0;
    k_normal_bf16<<<grid_for(count), 256, 0, s>>>(out, count, seed, start, sigma);
    return (int)cudaGetLastError();
}

}  // extern "C"
