// quantize.cu -- GPU round-to-nearest quantize/pack, the canonical <-> tiled
// layout conversion, and activation group sums.
//
// Quantize follows the page "Weight quantization" (tirogla.com), section
// "How it works" (scale/zero/q formulas) and section "Code" (function
// `quantize`): f32 throughout, IEEE division, ties away from zero, zero added
// after rounding, low nibble = even index.  This file is compiled with
// --fmad=false and every rounding step uses an explicit _rn intrinsic, so the
// codes, scales and zeros are bit-identical to the page's f32 arithmetic.
//
// The symmetric variant follows the page "Quantization" (hritesh-sonawane.
// github.io notes), sections "How it really works" and "Code" (int_quant):
// scale = max|w| / 7 (1 when that quotient is 0), q = clamp(round(w / scale),
// -8, 7) with ties to even, stored as code q + 8 with zero 8 in the same
// canonical arrays.
#include "common.cuh"

namespace q4 {

// Warp-wide minimum / maximum of one f32 per lane (exact selections;
// subnormal values come through unchanged -- groups made of subnormals
// quantize bit-identically to the oracle).
__device__ __forceinline__ float warp_min(float v)
{
    float r;
    asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
// Warp-wide maximum of one |w| per lane: for non-negative floats the bit
// patterns are ordered like the values.
__device__ __forceinline__ float warp_absmax(float a)
{
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;"
                 : "=r"(r)
                 : "r"(__float_as_uint(a) & 0x7fffffffu));
    return __uint_as_float(r);
}

// Code of one weight: clamp(round(w / s) + z, 0, 15) with the quotient of
// IEEE f32 division and ties away from zero, for |w / s| <= 16.
// The product qa = w * r with the rounded reciprocal r differs from the exact
// quotient by at most 2^-19 there (two roundings of relative 2^-24 on a value
// below 16), and the IEEE quotient by at most 2^-20.  Adding 1.5 * 2^23
// rounds qa to the nearest integer n (its bits minus those of 1.5 * 2^23 are
// n); when qa - n lies within 1/2 - 2^-16 of zero, both quotients round to n
// under any tie rule.  Otherwise (a quotient near n + 1/2, or a non-finite
// product) the division is done.
__device__ __forceinline__ int code_of(float w, float s, float r, int z)
{
    const float qa = __fmul_rn(w, r);
    const float t = __fadd_rn(qa, 12582912.0f);
    const float rem = __fsub_rn(qa, __fsub_rn(t, 12582912.0f));
    int q;
    if (fabsf(rem) < 0.5f - 0x1p-16f)  // false for NaN
        q = __float_as_int(t) - 0x4B400000;
    else
        q = static_cast<int>(roundf(__fdiv_rn(w, s)));
    q += z;
    return q < 0 ? 0 : (q > 15 ? 15 : q);
}

// Symmetric code: clamp(rint(w / s), -8, 7) + 8 with the IEEE f32 quotient
// and ties to even, for |w / s| <= 16.  Same reciprocal shortcut and
// fallback as code_of: away from a tie the rounded product names the
// quotient's integer under any tie rule.
__device__ __forceinline__ int code_sym(float w, float s, float r)
{
    const float qa = __fmul_rn(w, r);
    const float t = __fadd_rn(qa, 12582912.0f);
    const float rem = __fsub_rn(qa, __fsub_rn(t, 12582912.0f));
    int q;
    if (fabsf(rem) < 0.5f - 0x1p-16f)  // false for NaN
        q = __float_as_int(t) - 0x4B400000;
    else
        q = static_cast<int>(rintf(__fdiv_rn(w, s)));
    q = q < -8 ? -8 : (q > 7 ? 7 : q);
    return q + 8;
}

// One warp per group of 128 weights: each lane holds 4 consecutive weights
// (one 16-byte load), warp-wide min/max (exact, order-free), then every lane
// quantizes its 4 weights and stores 2 packed bytes.  A warp takes GPW groups
// per pass, loading all of them before computing (so that enough loads are
// in flight to keep HBM busy) and computing their scales in one go.
constexpr int GPW = 4;

template <bool SYM>
__global__ void __launch_bounds__(256) k_quantize(const float *__restrict__ w, int64_t ngroups,
                                                  uint8_t *__restrict__ packed,
                                                  float *__restrict__ scale,
                                                  uint8_t *__restrict__ zero, unsigned int *err)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t g0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * GPW;
         g0 < ngroups; g0 += nwarps * GPW) {
        float4 vv[GPW];
#pragma unroll
        for (int u = 0; u < GPW; ++u)
            vv[u] = g0 + u < ngroups ? __ldcs(reinterpret_cast<const float4 *>(w + (g0 + u) * G) + lane)
                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        // group ranges; then lane u (< GPW) computes group u's scale, zero
        // and reciprocal, once for all lanes, and broadcasts them
        float mys, myz;
        if constexpr (SYM) {
            float mya = 0.0f;
#pragma unroll
            for (int u = 0; u < GPW; ++u) {
                const float4 v = vv[u];
                const float a = warp_absmax(
                    fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                if (lane == u) mya = a;
            }
            mys = __fdiv_rn(mya, 7.0f);
            if (mys == 0.0f) mys = 1.0f;
            myz = 8.0f;
        } else {
            float mylo = 0.0f, myhi = 0.0f;
#pragma unroll
            for (int u = 0; u < GPW; ++u) {
                const float4 v = vv[u];
                const float lo = warp_min(fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
                const float hi = warp_max(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                if (lane == u) {
                    mylo = lo;
                    myhi = hi;
                }
            }
            // keep 0 exactly representable
            mylo = fminf(mylo, 0.0f);
            myhi = fmaxf(myhi, 0.0f);
            mys = (myhi > mylo) ? __fdiv_rn(__fsub_rn(myhi, mylo), 15.0f) : 1.0f;
            myz = fminf(fmaxf(roundf(__fdiv_rn(-mylo, mys)), 0.0f), 15.0f);
        }
        const float myr = __frcp_rn(mys);
#pragma unroll
        for (int u = 0; u < GPW; ++u) {
            const int64_t gi = g0 + u;
            if (gi >= ngroups) break;
            const float4 v = vv[u];
            const float sc = __shfl_sync(0xffffffffu, mys, u);
            const float r = __shfl_sync(0xffffffffu, myr, u);
            const int zi = static_cast<int>(__shfl_sync(0xffffffffu, myz, u));
            // flat index gi*128 + 4*lane + i: even index in the low nibble
            auto code = [&](float x) -> uint32_t {
                if constexpr (SYM) return static_cast<uint32_t>(code_sym(x, sc, r));
                else return static_cast<uint32_t>(code_of(x, sc, r, zi));
            };
            const uint32_t two =
                code(v.x) | (code(v.y) << 4) | (code(v.z) << 8) | (code(v.w) << 12);
            if (store_ok(gi * (G / 2) + 2 * lane, ngroups * (G / 2), err))
                reinterpret_cast<uint16_t *>(packed + gi * (G / 2))[lane] = static_cast<uint16_t>(two);
            if (lane == u && store_ok(gi, ngroups, err)) {
                scale[gi] = mys;
                zero[gi] = static_cast<uint8_t>(myz);
            }
        }
    }
}

// ---------------------------------------------------------------- tiled layout
// Word i of chunk c of lane l in tile (rt, g) covers k-step j = 4c+i, tile
// rows r = l/4 and r+8, and k offsets 16j + 2(l%4) + {0,1,8,9} inside group
// g.  Its eight nibble fields are filled from four canonical bytes (each byte
// holds an even/odd k pair):
//   B0 = (row r,   k0)     -> fields 0 (low nibble) and 16 (high nibble)
//   B1 = (row r+8, k0)     -> fields 4 and 20
//   B2 = (row r+8, k0 + 8) -> fields 8 and 24
//   B3 = (row r,   k0 + 8) -> fields 12 and 28
// with k0 = 16j + 2(l%4).  The low nibbles land in bits 0..15 and the high
// nibbles in bits 16..31, so one mask-and-or yields a pair of 16-bit values.
__device__ __forceinline__ uint32_t interleave4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3)
{
    const uint32_t lo = (b0 & 15u) | ((b1 & 15u) << 4) | ((b2 & 15u) << 8) | ((b3 & 15u) << 12);
    const uint32_t hi = (b0 >> 4) | ((b1 >> 4) << 4) | ((b2 >> 4) << 8) | ((b3 >> 4) << 12);
    return lo | (hi << 16);
}

// Code chunk `unit` (0..63) of tile (row0, g): 16 bytes, lane l = unit % 32,
// chunk c = unit / 32 (see the word layout above).
__device__ __forceinline__ uint4 code_chunk(const uint8_t *__restrict__ packed, int N, int K,
                                            int64_t row0, int g, int unit)
{
    const int c = unit >> 5, l = unit & 31;
    const int r = l >> 2, t = l & 3;
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * c + i;
        const int64_t kb = static_cast<int64_t>(g) * G + 16 * j + 2 * t;  // even k
        auto byte_at = [&](int64_t row, int64_t k) -> uint32_t {
            return row < N ? packed[row * (K / 2) + k / 2] : 0u;
        };
        out[i] = interleave4(byte_at(row0 + r, kb), byte_at(row0 + r + 8, kb),
                             byte_at(row0 + r + 8, kb + 8), byte_at(row0 + r, kb + 8));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// 69 sixteen-byte units per tile: 64 code chunks, 4 scale units, 1 zero unit.
__global__ void k_repack(const uint8_t *__restrict__ packed, const float *__restrict__ scale,
                         const uint8_t *__restrict__ zero, int N, int K, int64_t ntiles_total,
                         uint8_t *__restrict__ qw, unsigned int *err)
{
    const int NG = K / G;
    const int64_t units = ntiles_total * 69;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = u / 69;
        const int unit = static_cast<int>(u % 69);
        int64_t rt;
        int g;
        tile_of(tile, (N + TILE_ROWS - 1) / TILE_ROWS, NG, rt, g);
        const int64_t row0 = rt * TILE_ROWS;
        uint8_t *dst = qw + tile * TILE_BYTES;
        if (!store_ok(tile * TILE_BYTES + unit * 16 + 15, ntiles_total * TILE_BYTES, err)) continue;
        if (unit < 64) {
            *reinterpret_cast<uint4 *>(dst + unit * 16) = code_chunk(packed, N, K, row0, g, unit);
        } else if (unit < 68) {
            float sv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int pair = 2 * (unit - 64) + (e >> 1);  // pair index 0..7
                const int64_t row = row0 + pair + ((e & 1) ? 8 : 0);
                sv[e] = row < N ? scale[row * NG + g] : 0.0f;
            }
            *reinterpret_cast<float4 *>(dst + SCALE_OFF + (unit - 64) * 16) =
                make_float4(sv[0], sv[1], sv[2], sv[3]);
        } else {
            uint32_t zw[4] = {0, 0, 0, 0};
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const int pair = b >> 1;
                const int64_t row = row0 + pair + ((b & 1) ? 8 : 0);
                const uint32_t zv = row < N ? zero[row * NG + g] : 0u;
                zw[b >> 2] |= zv << ((b & 3) * 8);
            }
            *reinterpret_cast<uint4 *>(dst + ZERO_OFF) = make_uint4(zw[0], zw[1], zw[2], zw[3]);
        }
    }
}

// Compact tiles: 67 sixteen-byte units per tile: 64 code chunks, 2 units of
// binary16 scale pairs (each scale rounded to nearest even), 1 unit of 8
// zero-nibble pairs and 8 bytes of padding.
__global__ void k_repack_compact(const uint8_t *__restrict__ packed, const float *__restrict__ scale,
                                 const uint8_t *__restrict__ zero, int N, int K, int64_t ntiles_total,
                                 uint8_t *__restrict__ qw, unsigned int *err)
{
    const int NG = K / G;
    const int64_t units = ntiles_total * 67;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = u / 67;
        const int unit = static_cast<int>(u % 67);
        int64_t rt;
        int g;
        tile_of(tile, (N + TILE_ROWS - 1) / TILE_ROWS, NG, rt, g);
        const int64_t row0 = rt * TILE_ROWS;
        uint8_t *dst = qw + tile * CMP_TILE_BYTES;
        if (!store_ok(tile * CMP_TILE_BYTES + unit * 16 + 15, ntiles_total * CMP_TILE_BYTES, err))
            continue;
        if (unit < 64) {
            *reinterpret_cast<uint4 *>(dst + unit * 16) = code_chunk(packed, N, K, row0, g, unit);
        } else if (unit < 66) {
            uint32_t hw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {  // pair 4 (unit - 64) + e: rows pair, pair + 8
                const int pair = 4 * (unit - 64) + e;
                const int64_t r0 = row0 + pair, r8 = r0 + 8;
                const __half h0 = __float2half_rn(r0 < N ? scale[r0 * NG + g] : 0.0f);
                const __half h8 = __float2half_rn(r8 < N ? scale[r8 * NG + g] : 0.0f);
                hw[e] = static_cast<uint32_t>(__half_as_ushort(h0)) |
                        (static_cast<uint32_t>(__half_as_ushort(h8)) << 16);
            }
            *reinterpret_cast<uint4 *>(dst + SCALE_OFF + (unit - 64) * 16) =
                make_uint4(hw[0], hw[1], hw[2], hw[3]);
        } else {
            uint32_t zw[2] = {0, 0};
#pragma unroll
            for (int b = 0; b < 8; ++b) {  // pair b: rows b (low nibble), b + 8 (high)
                const int64_t r0 = row0 + b, r8 = r0 + 8;
                const uint32_t z0 = r0 < N ? (zero[r0 * NG + g] & 15u) : 0u;
                const uint32_t z8 = r8 < N ? (zero[r8 * NG + g] & 15u) : 0u;
                zw[b >> 2] |= (z0 | (z8 << 4)) << ((b & 3) * 8);
            }
            *reinterpret_cast<uint4 *>(dst + CMP_ZERO_OFF) = make_uint4(zw[0], zw[1], 0u, 0u);
        }
    }
}

// Code word i of chunk c of lane l of tile (row0, g) back into the
// canonical bytes (rows past N are dropped).
__device__ __forceinline__ void put_code_word(uint8_t *__restrict__ packed, int N, int K,
                                              int64_t row0, int g, int c, int l, int i, uint32_t w,
                                              unsigned int *err)
{
    const int r = l >> 2, t = l & 3, j = 4 * c + i;
    const int64_t kb = static_cast<int64_t>(g) * G + 16 * j + 2 * t;
    auto put = [&](int64_t row, int64_t k, int f) {
        if (row < N && store_ok(row * (K / 2) + k / 2, static_cast<int64_t>(N) * (K / 2), err)) {
            const uint32_t lo = (w >> (4 * f)) & 15u, hi = (w >> (16 + 4 * f)) & 15u;
            packed[row * (K / 2) + k / 2] = static_cast<uint8_t>(lo | (hi << 4));
        }
    };
    put(row0 + r, kb, 0);
    put(row0 + r + 8, kb, 1);
    put(row0 + r + 8, kb + 8, 2);
    put(row0 + r, kb + 8, 3);
}

// Inverse: one thread per code word (4 canonical bytes), plus one per tile
// row-pair for the metadata.
__global__ void k_unpack(const uint8_t *__restrict__ qw, int N, int K, int64_t ntiles_total,
                         uint8_t *__restrict__ packed, float *__restrict__ scale,
                         uint8_t *__restrict__ zero, unsigned int *err)
{
    const int NG = K / G;
    const int64_t units = ntiles_total * (256 + 8);
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = u / 264;
        const int unit = static_cast<int>(u % 264);
        int64_t rt;
        int g;
        tile_of(tile, (N + TILE_ROWS - 1) / TILE_ROWS, NG, rt, g);
        const int64_t row0 = rt * TILE_ROWS;
        const uint8_t *src = qw + tile * TILE_BYTES;
        if (unit < 256) {
            const int c = unit >> 7, l = (unit >> 2) & 31, i = unit & 3;
            const uint32_t w = reinterpret_cast<const uint32_t *>(src)[(c * 32 + l) * 4 + i];
            put_code_word(packed, N, K, row0, g, c, l, i, w, err);
        } else {
            const int pair = unit - 256;
            const float *sp = reinterpret_cast<const float *>(src + SCALE_OFF) + 2 * pair;
            const uint8_t *zp = src + ZERO_OFF + 2 * pair;
            const int64_t lim = static_cast<int64_t>(N) * NG;
            if (row0 + pair < N && store_ok((row0 + pair) * NG + g, lim, err)) {
                scale[(row0 + pair) * NG + g] = sp[0];
                zero[(row0 + pair) * NG + g] = zp[0];
            }
            if (row0 + pair + 8 < N && store_ok((row0 + pair + 8) * NG + g, lim, err)) {
                scale[(row0 + pair + 8) * NG + g] = sp[1];
                zero[(row0 + pair + 8) * NG + g] = zp[1];
            }
        }
    }
}

// Inverse of the compact layout: codes, binary16 scale bits, one zero byte
// per group.
__global__ void k_unpack_compact(const uint8_t *__restrict__ qw, int N, int K, int64_t ntiles_total,
                                 uint8_t *__restrict__ packed, uint16_t *__restrict__ scale16,
                                 uint8_t *__restrict__ zero, unsigned int *err)
{
    const int NG = K / G;
    const int64_t units = ntiles_total * (256 + 8);
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = u / 264;
        const int unit = static_cast<int>(u % 264);
        int64_t rt;
        int g;
        tile_of(tile, (N + TILE_ROWS - 1) / TILE_ROWS, NG, rt, g);
        const int64_t row0 = rt * TILE_ROWS;
        const uint8_t *src = qw + tile * CMP_TILE_BYTES;
        if (unit < 256) {
            const int c = unit >> 7, l = (unit >> 2) & 31, i = unit & 3;
            const uint32_t w = reinterpret_cast<const uint32_t *>(src)[(c * 32 + l) * 4 + i];
            put_code_word(packed, N, K, row0, g, c, l, i, w, err);
        } else {
            const int pair = unit - 256;
            const uint16_t *sp = reinterpret_cast<const uint16_t *>(src + SCALE_OFF) + 2 * pair;
            const uint32_t zb = src[CMP_ZERO_OFF + pair];
            const int64_t lim = static_cast<int64_t>(N) * NG;
            if (row0 + pair < N && store_ok((row0 + pair) * NG + g, lim, err)) {
                scale16[(row0 + pair) * NG + g] = sp[0];
                zero[(row0 + pair) * NG + g] = static_cast<uint8_t>(zb & 15u);
            }
            if (row0 + pair + 8 < N && store_ok((row0 + pair + 8) * NG + g, lim, err)) {
                scale16[(row0 + pair + 8) * NG + g] = sp[1];
                zero[(row0 + pair + 8) * NG + g] = static_cast<uint8_t>(zb >> 4);
            }
        }
    }
}

// Activation group sums: one warp per (m, g), f32 accumulation.
__global__ void k_xsum(const void *__restrict__ x, q4_dtype xt, int64_t M, int64_t K,
                       float *__restrict__ xsum, unsigned int *err)
{
    const int lane = threadIdx.x & 31;
    const int64_t NG = K / G, total = M * NG;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         id < total; id += nwarps) {
        const int64_t m = id / NG, g = id % NG;
        const int64_t base = m * K + g * G + 4 * lane;
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) s += load_x_f32(x, xt, base + i);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0 && store_ok(id, total, err)) xsum[id] = s;
    }
}

static int grid_for(int64_t work, int threads)
{
    int64_t b = (work + threads - 1) / threads;
    const int64_t cap = 152LL * 32;
    if (b > cap) b = cap;
    return static_cast<int>(b < 1 ? 1 : b);
}

cudaError_t quantize_launch(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                            uint8_t *zero, bool symmetric, unsigned int *err, cudaStream_t s)
{
    const int64_t ngroups = N * K / G;
    const int grid = grid_for((ngroups + GPW - 1) / GPW * 32, 256);
    if (symmetric)
        k_quantize<true><<<grid, 256, 0, s>>>(w, ngroups, packed, scale, zero, err);
    else
        k_quantize<false><<<grid, 256, 0, s>>>(w, ngroups, packed, scale, zero, err);
    return cudaGetLastError();
}

cudaError_t repack_launch(const uint8_t *packed, const float *scale, const uint8_t *zero,
                          int64_t N, int64_t K, uint8_t *qw, unsigned int *err, cudaStream_t s)
{
    const int64_t ntiles = ((N + TILE_ROWS - 1) / TILE_ROWS) * (K / G);
    k_repack<<<grid_for(ntiles * 69, 256), 256, 0, s>>>(packed, scale, zero, static_cast<int>(N),
                                                        static_cast<int>(K), ntiles, qw, err);
    return cudaGetLastError();
}

cudaError_t unpack_launch(const uint8_t *qw, int64_t N, int64_t K, uint8_t *packed, float *scale,
                          uint8_t *zero, unsigned int *err, cudaStream_t s)
{
    const int64_t ntiles = ((N + TILE_ROWS - 1) / TILE_ROWS) * (K / G);
    k_unpack<<<grid_for(ntiles * 264, 256), 256, 0, s>>>(qw, static_cast<int>(N),
                                                         static_cast<int>(K), ntiles, packed,
                                                         scale, zero, err);
    return cudaGetLastError();
}

cudaError_t repack_compact_launch(const uint8_t *packed, const float *scale, const uint8_t *zero,
                                  int64_t N, int64_t K, uint8_t *qw, unsigned int *err,
                                  cudaStream_t s)
{
    const int64_t ntiles = ((N + TILE_ROWS - 1) / TILE_ROWS) * (K / G);
    k_repack_compact<<<grid_for(ntiles * 67, 256), 256, 0, s>>>(
        packed, scale, zero, static_cast<int>(N), static_cast<int>(K), ntiles, qw, err);
    return cudaGetLastError();
}

cudaError_t unpack_compact_launch(const uint8_t *qw, int64_t N, int64_t K, uint8_t *packed,
                                  uint16_t *scale16, uint8_t *zero, unsigned int *err,
                                  cudaStream_t s)
{
    const int64_t ntiles = ((N + TILE_ROWS - 1) / TILE_ROWS) * (K / G);
    k_unpack_compact<<<grid_for(ntiles * 264, 256), 256, 0, s>>>(
        qw, static_cast<int>(N), static_cast<int>(K), ntiles, packed, scale16, zero, err);
    return cudaGetLastError();
}

cudaError_t xsum_launch(const void *x, q4_dtype xt, int64_t M, int64_t K, float *xsum,
                        unsigned int *err, cudaStream_t s)
{
    const int64_t total = M * (K / G);
    k_xsum<<<grid_for(total * 32, 256), 256, 0, s>>>(x, xt, M, K, xsum, err);
    return cudaGetLastError();
}

}  // namespace q4
