// gemv.cu -- decode W4A16 GEMV for 1 <= M <= 16 on sm_103a.
//
// Computes y[m][n] = sum over groups g of
//     scale[n][g] * (sum_{k in g} q[n][k] * x[m][k] - zero[n][g] * sum_{k in g} x[m][k])
// i.e. the factored group dot of the page "Weight quantization" (tirogla.com,
// sections "How it works" and "Code", function `dot`), with the 4-bit codes
// turned into floating point in registers and never written back to memory.
//
// Structure (one CTA = 4 consumer warps + 1 producer warp):
//   * the CTA owns RB = 4 row tiles (64 output rows) and one slice of groups
//     along K; the producer warp streams the weight tiles of that block with
//     1-D bulk asynchronous copies (TMA engine) into a 3-stage shared-memory
//     ring, each stage holding RB row tiles x 4 consecutive groups;
//   * consumer warp w takes group w of every stage, keeps the activation
//     material for that group in registers and sweeps the RB tiles;
//   * partial sums are reduced across warps in shared memory and, when K is
//     split over several CTAs, across slices through a workspace, by the last
//     CTA of the row block to arrive (fixed summation order, so results do not
//     depend on timing).
//
// Two consumer variants:
//   FMA (M = 1): CUDA-core path.  A 4-bit code q at bit offset 16 or 12 of a
//     word becomes the f32 value 1 + q/128 or 1 + q/2048 with one LOP3
//     (mantissa bits, exponent of 1.0); two such values are multiplied into a
//     pair of f32 accumulators by one packed FFMA2.  The constant 1 is removed
//     per group with the pre-computed activation sums.
//   MMA (M = 1..16, bf16/f16 activations; f32 activations split into bf16
//     hi + lo): each word yields the four A-fragment registers of an
//     m16n8k16 tensor-core MMA as bf16 pairs 128 + q (f16: 1024 + q) with one
//     LOP3 each; the activations are the B fragment (the batch is the MMA's
//     n dimension); per group, y += scale * (D - (offset + zero) * sum x).
#include "common.cuh"

namespace q4 {

constexpr int W = 4;        // consumer warps
constexpr int RB = 4;       // row tiles per CTA
constexpr int NSTAGE = 3;   // ring depth
constexpr int THREADS = (W + 1) * 32;
constexpr int STAGE_BYTES = RB * W * TILE_BYTES;  // 17664
constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;  // 52992
constexpr int CTRL_BYTES = 128;                   // barriers + flags
constexpr int GS_MAX_FMA = 16;
constexpr int GS_MAX_MMA = 32;
constexpr int FMA_XP_FLOATS = 4 * 8 * 8;  // per group: 4 lane classes x 8 words x 8 floats

static_assert(RING_BYTES % 128 == 0, "ring alignment");
static_assert(W * RB * 16 * 16 * 4 <= RING_BYTES, "reduction buffer fits in the ring");

__host__ __device__ constexpr int smem_bytes(int mode)
{
    return RING_BYTES + CTRL_BYTES +
           (mode == PATH_FMA ? GS_MAX_FMA * (FMA_XP_FLOATS + 16) * 4 : GS_MAX_MMA * 16 * 4);
}

__device__ __forceinline__ void store_y(void *y, q4_dtype yt, int64_t idx, float v)
{
    if (yt == Q4_F32)
        static_cast<float *>(y)[idx] = v;
    else if (yt == Q4_BF16)
        static_cast<__nv_bfloat16 *>(y)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half *>(y)[idx] = __float2half_rn(v);
}

// (1 + q_hi/128, 1 + q_lo/2048) from the codes at bit offsets 16 and 12.
__device__ __forceinline__ float2 code_pair(uint32_t v)
{
    return make_float2(__uint_as_float(lop3_and_or(v, 0x000F0000u, 0x3F800000u)),
                       __uint_as_float(lop3_and_or(v, 0x0000F000u, 0x3F800000u)));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ABT: 0 = bf16 operands (magic 128 + q), 1 = f16 operands (magic 1024 + q).
// XSPLIT: f32 activations carried as bf16 hi + bf16 lo (two MMAs per step).
template <int MODE, int NT, int ABT, bool XSPLIT>
__global__ void __launch_bounds__(THREADS) k_gemv(const GemvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint64_t *empty = full + NSTAGE;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NSTAGE);
    int *last_flag = reinterpret_cast<int *>(empty + NSTAGE) + 1;
    float *xmat = reinterpret_cast<float *>(smem + RING_BYTES + CTRL_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = a.K / G;
    const int ntiles = (a.N + TILE_ROWS - 1) / TILE_ROWS;
    const int ks = blockIdx.x % a.ks;
    const int rb = blockIdx.x / a.ks;
    const int rt0 = rb * RB;
    const int nrt = min(RB, ntiles - rt0);
    const int g_begin = ks * a.gs;
    const int g_end = min(NG, g_begin + a.gs);
    const int nsteps = (g_end - g_begin + W - 1) / W;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == W) {
        if (lane == 0) {
            int issued = 0;
            if (!a.debug_no_copy) {
                for (int s = 0; s < nsteps; ++s) {
                    const int slot = s % NSTAGE;
                    if (s >= NSTAGE &&
                        !mbar_wait_bounded(&empty[slot], ((s / NSTAGE) - 1) & 1, abort_flag,
                                           a.wait_ns, a.err))
                        break;
                    const int g0 = g_begin + s * W;
                    const int ng = min(W, g_end - g0);
                    const uint32_t row_bytes = static_cast<uint32_t>(ng) * TILE_BYTES;
                    mbar_arrive_expect_tx(&full[slot], row_bytes * nrt);
                    for (int r = 0; r < nrt; ++r) {
                        const uint8_t *src =
                            a.qw + (static_cast<int64_t>(rt0 + r) * NG + g0) * TILE_BYTES;
                        bulk_g2s(ring + slot * STAGE_BYTES + r * W * TILE_BYTES, src, row_bytes,
                                 &full[slot]);
                    }
                    ++issued;
                }
            }
            // Every issued copy must land before the CTA may exit.
            for (int s = max(0, issued - NSTAGE); s < issued; ++s)
                mbar_wait_bounded(&full[s % NSTAGE], (s / NSTAGE) & 1, abort_flag, a.wait_ns,
                                  a.err, false);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int gq = lane >> 2, t = lane & 3;
    const int ngs = g_end - g_begin;
    const int M = a.M;

    if (MODE == PATH_FMA) {
        // Activation pairs in the order the code fields are extracted (see
        // the word layout in q4.h): per word, (x1,x8) (x9,x1) (x8,x0)
        // (x0',x9) with xa = x[16j + 2t + a] and x0' from the next word of
        // the same 16-byte chunk; plus S = sum x and the two offset terms.
        float *xp = xmat;
        float4 *xs = reinterpret_cast<float4 *>(xmat + GS_MAX_FMA * FMA_XP_FLOATS);
        for (int rec = threadIdx.x; rec < ngs * 4; rec += W * 32) {
            const int gl = rec >> 2, tt = rec & 3;
            const int64_t kg = static_cast<int64_t>(g_begin + gl) * G + 2 * tt;
            float slo = 0.0f, shi = 0.0f;
            float4 *dst = reinterpret_cast<float4 *>(xp + rec * 64);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int jn = (j & 4) | ((j + 1) & 3);
                const float x0 = load_x_f32(a.x, a.xt, kg + 16 * j);
                const float x1 = load_x_f32(a.x, a.xt, kg + 16 * j + 1);
                const float x8 = load_x_f32(a.x, a.xt, kg + 16 * j + 8);
                const float x9 = load_x_f32(a.x, a.xt, kg + 16 * j + 9);
                const float x0n = load_x_f32(a.x, a.xt, kg + 16 * jn);
                dst[2 * j] = make_float4(x1, x8, x9, x1);
                dst[2 * j + 1] = make_float4(x8, x0, x0n, x9);
                slo += x0 + x1;
                shi += x8 + x9;
            }
            xs[rec] = make_float4(slo + shi, 128.0f * slo + 2048.0f * shi,
                                  128.0f * shi + 2048.0f * slo, 0.0f);
        }
    } else {
        float *sx = xmat;  // [gl][16]
        for (int id = threadIdx.x; id < ngs * M; id += W * 32) {
            const int gl = id / M, m = id % M;
            const int64_t base = static_cast<int64_t>(m) * a.K + static_cast<int64_t>(g_begin + gl) * G;
            float s = 0.0f;
            for (int i = 0; i < G; ++i) s += load_x_f32(a.x, a.xt, base + i);
            sx[gl * 16 + m] = s;
        }
    }
    named_barrier_sync(1, W * 32);

    float yacc[RB][NT][4];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) yacc[r][n][e] = 0.0f;

    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
        const int slot = s % NSTAGE;
        const int g = g_begin + s * W + warp;
        ok = mbar_wait_bounded(&full[slot], (s / NSTAGE) & 1, abort_flag, a.wait_ns, a.err);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (g < g_end) {
            const int gl = g - g_begin;
            const uint8_t *stage = ring + slot * STAGE_BYTES + warp * TILE_BYTES;
            if (MODE == PATH_FMA) {
                const float4 *xpp = reinterpret_cast<const float4 *>(xmat + (gl * 4 + t) * 64);
                float2 P[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 u = xpp[2 * j], v = xpp[2 * j + 1];
                    P[j][0] = make_float2(u.x, u.y);
                    P[j][1] = make_float2(u.z, u.w);
                    P[j][2] = make_float2(v.x, v.y);
                    P[j][3] = make_float2(v.z, v.w);
                }
                const float4 xsv =
                    reinterpret_cast<const float4 *>(xmat + GS_MAX_FMA * FMA_XP_FLOATS)[gl * 4 + t];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    if (r < nrt) {
                        const uint8_t *tile = stage + r * W * TILE_BYTES;
                        const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                        const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane);
                        const float2 sp = *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq);
                        const uint32_t zp = *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq);
                        const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        float2 accG = make_float2(0.0f, 0.0f), accG8 = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t wj = wv[j], wn = wv[(j & 4) | ((j + 1) & 3)];
                            accG = __ffma2_rn(code_pair(wj), P[j][0], accG);
                            accG8 = __ffma2_rn(code_pair(wj >> 8), P[j][1], accG8);
                            accG8 = __ffma2_rn(code_pair(wj << 8), P[j][2], accG8);
                            accG = __ffma2_rn(code_pair(__funnelshift_r(wj, wn, 16)), P[j][3], accG);
                        }
                        const float zg = static_cast<float>(zp & 0xFFu);
                        const float zg8 = static_cast<float>(zp >> 8);
                        const float ig =
                            fmaf(128.0f, accG.x, fmaf(2048.0f, accG.y, -fmaf(zg, xsv.x, xsv.y)));
                        const float ig8 =
                            fmaf(128.0f, accG8.x, fmaf(2048.0f, accG8.y, -fmaf(zg8, xsv.x, xsv.z)));
                        yacc[r][0][0] = fmaf(sp.x, ig, yacc[r][0][0]);
                        yacc[r][0][2] = fmaf(sp.y, ig8, yacc[r][0][2]);
                    }
                }
            } else {
                // B fragments of this group for every n-tile (batch rows 8n + gq)
                uint32_t bh[NT][8][2], bl[XSPLIT ? NT : 1][8][2];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int m = 8 * n + gq;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int64_t k = static_cast<int64_t>(g) * G + 16 * j + 2 * t;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t vh = 0, vl = 0;
                            if (m < M) {
                                const int64_t idx = static_cast<int64_t>(m) * a.K + k + 8 * h;
                                if (XSPLIT) {
                                    const float2 xv = *reinterpret_cast<const float2 *>(
                                        static_cast<const float *>(a.x) + idx);
                                    vh = pack_bf16x2(xv.x, xv.y);
                                    vl = pack_bf16x2(xv.x - bf16_lo_f32(vh), xv.y - bf16_hi_f32(vh));
                                } else {
                                    vh = *reinterpret_cast<const uint32_t *>(
                                        static_cast<const uint16_t *>(a.x) + idx);
                                }
                            }
                            bh[n][j][h] = vh;
                            if (XSPLIT) bl[XSPLIT ? n : 0][j][h] = vl;
                        }
                    }
                }
                const uint32_t MAG = ABT == 0 ? 0x43004300u : 0x64006400u;
                const float OFF = ABT == 0 ? 128.0f : 1024.0f;
                float S0[NT], S1[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    S0[n] = xmat[gl * 16 + 8 * n + 2 * t];
                    S1[n] = xmat[gl * 16 + 8 * n + 2 * t + 1];
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    if (r < nrt) {
                        const uint8_t *tile = stage + r * W * TILE_BYTES;
                        const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                        const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane);
                        const float2 sp = *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq);
                        const uint32_t zp = *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq);
                        const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        float d[NT][4];
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) d[n][e] = 0.0f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t w = wv[j];
                            const uint32_t a0 = lop3_and_or(w, 0x000F000Fu, MAG);
                            const uint32_t a1 = lop3_and_or(w >> 4, 0x000F000Fu, MAG);
                            const uint32_t a3 = lop3_and_or(w >> 8, 0x000F000Fu, MAG);
                            const uint32_t a2 = lop3_and_or(w >> 12, 0x000F000Fu, MAG);
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                if (ABT == 0) {
                                    mma_bf16(d[n], a0, a1, a2, a3, bh[n][j][0], bh[n][j][1]);
                                    if (XSPLIT)
                                        mma_bf16(d[n], a0, a1, a2, a3, bl[XSPLIT ? n : 0][j][0],
                                                 bl[XSPLIT ? n : 0][j][1]);
                                } else {
                                    mma_f16(d[n], a0, a1, a2, a3, bh[n][j][0], bh[n][j][1]);
                                }
                            }
                        }
                        const float zg = OFF + static_cast<float>(zp & 0xFFu);
                        const float zg8 = OFF + static_cast<float>(zp >> 8);
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            yacc[r][n][0] = fmaf(sp.x, fmaf(-zg, S0[n], d[n][0]), yacc[r][n][0]);
                            yacc[r][n][1] = fmaf(sp.x, fmaf(-zg, S1[n], d[n][1]), yacc[r][n][1]);
                            yacc[r][n][2] = fmaf(sp.y, fmaf(-zg8, S0[n], d[n][2]), yacc[r][n][2]);
                            yacc[r][n][3] = fmaf(sp.y, fmaf(-zg8, S1[n], d[n][3]), yacc[r][n][3]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------------- reduction and output
    named_barrier_sync(1, W * 32);
    if (*abort_flag) return;  // timed out: write nothing

    // All copies have been consumed, so the ring is free: red[w][row][m]
    float *red = reinterpret_cast<float *>(ring);
    const int MS = (MODE == PATH_FMA) ? 1 : 16;
    if (MODE == PATH_FMA) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float v = yacc[r][0][0], v8 = yacc[r][0][2];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v8 += __shfl_xor_sync(0xffffffffu, v8, 1);
            v8 += __shfl_xor_sync(0xffffffffu, v8, 2);
            if (t == 0) {
                red[(warp * RB * 16 + r * 16 + gq) * MS] = v;
                red[(warp * RB * 16 + r * 16 + gq + 8) * MS] = v8;
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = r * 16 + gq + ((e & 2) ? 8 : 0);
                    const int m = 8 * n + 2 * t + (e & 1);
                    red[(warp * RB * 16 + row) * MS + m] = yacc[r][n][e];
                }
    }
    named_barrier_sync(1, W * 32);

    const int Mo = (MODE == PATH_FMA) ? 1 : M;
    const int npad = ntiles * TILE_ROWS;
    const int nout = nrt * 16 * Mo;
    const int row0 = rt0 * TILE_ROWS;
    for (int i = threadIdx.x; i < nout; i += W * 32) {
        const int row = i / Mo, m = i % Mo;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) v += red[(w * RB * 16 + row) * MS + m];
        if (a.ks == 1) {
            if (row0 + row < a.N) store_y(a.y, a.yt, static_cast<int64_t>(m) * a.N + row0 + row, v);
        } else {
            a.partial[(static_cast<int64_t>(ks) * M + m) * npad + row0 + row] = v;
        }
    }
    if (a.ks == 1) return;

    // Split over K: the last CTA of this row block sums the slices in order.
    __threadfence();
    named_barrier_sync(1, W * 32);
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(&a.count[rb], 1u);
        *last_flag = (prev == static_cast<unsigned int>(a.ks - 1));
    }
    named_barrier_sync(1, W * 32);
    if (!*last_flag) return;
    __threadfence();
    for (int i = threadIdx.x; i < nout; i += W * 32) {
        const int row = i / Mo, m = i % Mo;
        if (row0 + row >= a.N) continue;
        float v = 0.0f;
        for (int s2 = 0; s2 < a.ks; ++s2)
            v += __ldcg(&a.partial[(static_cast<int64_t>(s2) * M + m) * npad + row0 + row]);
        store_y(a.y, a.yt, static_cast<int64_t>(m) * a.N + row0 + row, v);
    }
    if (threadIdx.x == 0) a.count[rb] = 0u;  // ready for the next call
}

// -------------------------------------------------------------------- host
template <int MODE, int NT, int ABT, bool XSPLIT>
static cudaError_t launch_one(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = k_gemv<MODE, NT, ABT, XSPLIT>;
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes(MODE));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int grid = p.nrb * p.ks;
    kern<<<grid, THREADS, smem_bytes(MODE), s>>>(a);
    return cudaGetLastError();
}

size_t counters_bytes(int nrb)
{
    return ((static_cast<size_t>(nrb) * sizeof(unsigned int) + 255) / 256) * 256;
}

GemvPlan gemv_plan(int M, int N, int K, q4_dtype xt, int path, int sm_count)
{
    GemvPlan p{};
    if (path == PATH_AUTO) path = (M == 1) ? PATH_FMA : PATH_MMA;
    p.path = path;
    p.rb = RB;
    const int ntiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int NG = K / G;
    p.nrb = (ntiles + RB - 1) / RB;
    const int gs_max = (path == PATH_FMA) ? GS_MAX_FMA : GS_MAX_MMA;
    // Expected resident CTAs per SM (shared memory bound).
    const int per_sm = (path == PATH_FMA) ? 2 : 3;
    const long slots = static_cast<long>(sm_count) * per_sm;
    long best_cost = -1;
    int best_ks = 1, best_gs = NG;
    for (int gs = (NG < gs_max ? NG : gs_max); gs >= 1; --gs) {
        const int ks = (NG + gs - 1) / gs;
        const long units = static_cast<long>(p.nrb) * ks;
        const long waves = (units + slots - 1) / slots;
        // cost in group-steps: per-CTA work (gs groups + fixed overhead of
        // about 2) per wave, plus the split-K fixup.
        const long cost = waves * (gs + 2) * 4 + (ks > 1 ? 2 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_ks = ks;
            best_gs = gs;
        }
        if (gs < 4 && best_cost >= 0 && gs < best_gs) break;
    }
    p.ks = best_ks;
    p.gs = best_gs;
    if (p.ks > 1) {
        // [arrival counters, one per row block, padded to 256 B][partials]
        const size_t part = static_cast<size_t>(p.ks) * M * ntiles * TILE_ROWS * sizeof(float);
        p.workspace = counters_bytes(p.nrb) + part;
    } else {
        p.workspace = 0;
    }
    (void)xt;
    return p;
}

cudaError_t gemv_launch(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    if (p.path == PATH_FMA) return launch_one<PATH_FMA, 1, 0, false>(p, a, s);
    const int nt = a.M <= 8 ? 1 : 2;
    if (a.xt == Q4_F16)
        return nt == 1 ? launch_one<PATH_MMA, 1, 1, false>(p, a, s)
                       : launch_one<PATH_MMA, 2, 1, false>(p, a, s);
    if (a.xt == Q4_BF16)
        return nt == 1 ? launch_one<PATH_MMA, 1, 0, false>(p, a, s)
                       : launch_one<PATH_MMA, 2, 0, false>(p, a, s);
    return nt == 1 ? launch_one<PATH_MMA, 1, 0, true>(p, a, s)
                   : launch_one<PATH_MMA, 2, 0, true>(p, a, s);
}

}  // namespace q4
