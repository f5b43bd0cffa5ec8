// gemv.cu -- decode W4A16 GEMV for 1 <= M <= 16 on sm_103a.
//
// Computes y[m][n] = sum over groups g of
//     scale[n][g] * (sum_{k in g} q[n][k] * x[m][k] - zero[n][g] * sum_{k in g} x[m][k])
// i.e. the factored group dot of the page "Weight quantization" (tirogla.com,
// sections "How it works" and "Code", function `dot`), with the 4-bit codes
// turned into floating point in registers and never written back to memory.
//
// Structure: a persistent kernel, one CTA = 4 consumer warps + 1 producer
// warp, a few CTAs per SM.  The work is cut into units of RB = 4 row tiles
// (64 output rows) by one slice of groups along K; CTA c takes units c,
// c + grid, c + 2*grid, ...  The producer warp walks the same sequence and
// streams, with 1-D bulk asynchronous copies (TMA engine), the weight tiles
// into a 4-stage shared-memory ring (stage = RB row tiles x 4 consecutive
// groups) -- it runs ahead across unit boundaries, so the memory pipeline
// never drains between units.  Consumer warp w takes group w of every stage.
// Partial sums are reduced across warps in shared memory and, when K is split
// over several units, across slices through a workspace by the last unit of
// the row block to finish (fixed summation order: results do not depend on
// timing).
//
// Two consumer variants:
//   FMA (M = 1): CUDA-core path.  A 4-bit code q at bit offset 16 or 12 of a
//     word becomes the f32 value 1 + q/128 or 1 + q/2048 with one LOP3
//     (mantissa bits under the exponent of 1.0); two such values are
//     multiplied into a pair of f32 accumulators by one packed FFMA2.  The
//     constant 1 is removed per group with the activation sums.  The
//     producer also copies each unit's activation slice into a double-buffered
//     shared-memory slot; the consumers turn it into the per-lane pair order
//     once per unit.
//   MMA (M = 1..16, bf16/f16 activations; f32 activations as bf16 hi + lo):
//     each word yields the four A-fragment registers of an m16n8k16
//     tensor-core MMA as bf16 pairs 128 + q (f16: 1024 + q) with one LOP3
//     each; the activations are the B fragment (the batch is the MMA's n
//     dimension).  The group sums of the activations come from one extra MMA
//     per k-step with an all-ones A operand, once per group.  Per group,
//     y += scale * (D - (offset + zero) * sum x).
#include "common.cuh"

namespace q4 {

constexpr int W = 4;        // consumer warps
constexpr int RB = 4;       // row tiles per unit
constexpr int NSTAGE = 3;   // ring depth
constexpr int THREADS = (W + 1) * 32;
constexpr int CONSUMERS = W * 32;
constexpr int STAGE_BYTES = RB * W * TILE_BYTES;  // 17664
constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;  // 52992
constexpr int CTRL_BYTES = 128;                   // barriers + flags
constexpr int GS_MAX_FMA = 8;
constexpr int GS_MAX_MMA = 32;
// FMA activation pairs: one record of 64 floats per (group, lane class t),
// padded to 68 floats so the four lane classes of a warp read four different
// bank groups in the same wavefront.
constexpr int PAIR_STRIDE = 68;
constexpr int FMA_XSLOT_BYTES = GS_MAX_FMA * G * 4;  // one unit's activations (f32 worst case)
constexpr int FMA_PAIR_FLOATS = GS_MAX_FMA * 4 * PAIR_STRIDE;
constexpr int FMA_PAIR_BYTES = FMA_PAIR_FLOATS * 4 + GS_MAX_FMA * 4 * 16;
constexpr int RED_FLOATS_FMA = W * RB * 16;
constexpr int RED_FLOATS_MMA = W * RB * 16 * 16;
constexpr int MIN_BLOCKS = 3;  // CTAs per SM the shared memory budget is sized for

static_assert(RING_BYTES % 128 == 0, "ring alignment");
static_assert(MIN_BLOCKS * (RING_BYTES + CTRL_BYTES + 2 * FMA_XSLOT_BYTES + FMA_PAIR_BYTES +
                            RED_FLOATS_FMA * 4 + 1024) <= 228 * 1024,
              "three FMA CTAs per SM");
static_assert(MIN_BLOCKS * (RING_BYTES + CTRL_BYTES + RED_FLOATS_MMA * 4 + 1024) <= 228 * 1024,
              "three MMA CTAs per SM");

__host__ __device__ constexpr int smem_bytes(int mode)
{
    return mode == PATH_FMA
               ? RING_BYTES + CTRL_BYTES + 2 * FMA_XSLOT_BYTES + FMA_PAIR_BYTES + RED_FLOATS_FMA * 4
               : RING_BYTES + CTRL_BYTES + RED_FLOATS_MMA * 4;
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
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int ABT>
__device__ __forceinline__ void mma_ab(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1)
{
    if (ABT == 0)
        mma_bf16(d, a0, a1, a2, a3, b0, b1);
    else
        mma_f16(d, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float smem_x_f32(const uint8_t *xs, q4_dtype xt, int i)
{
    if (xt == Q4_F32) return reinterpret_cast<const float *>(xs)[i];
    const uint16_t b = reinterpret_cast<const uint16_t *>(xs)[i];
    if (xt == Q4_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
    __half_raw hr;
    hr.x = b;
    return __half2float(__half(hr));
}

struct UnitInfo {
    int rb, ks, rt0, nrt, g_begin, g_end, nsteps;
};

__device__ __forceinline__ UnitInfo unit_info(const GemvArgs &a, int u, int ntiles, int NG)
{
    UnitInfo ui;
    ui.ks = u % a.ks;
    ui.rb = u / a.ks;
    ui.rt0 = ui.rb * RB;
    ui.nrt = min(RB, ntiles - ui.rt0);
    ui.g_begin = ui.ks * a.gs;
    ui.g_end = min(NG, ui.g_begin + a.gs);
    ui.nsteps = (ui.g_end - ui.g_begin + W - 1) / W;
    return ui;
}

// ABT: 0 = bf16 operands (magic 128 + q), 1 = f16 operands (magic 1024 + q).
// XSPLIT: f32 activations carried as bf16 hi + bf16 lo (two MMAs per step).
template <int MODE, int NT, int ABT, bool XSPLIT>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS) k_gemv(const GemvArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint64_t *empty = full + NSTAGE;
    uint64_t *xfull = empty + NSTAGE;  // FMA activation slots
    uint64_t *xempty = xfull + 2;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(xempty + 2);
    int *last_flag = const_cast<int *>(abort_flag) + 1;
    uint8_t *after = smem + RING_BYTES + CTRL_BYTES;
    uint8_t *xslot = after;                                                 // FMA: 2 slots
    float *pairs = reinterpret_cast<float *>(after + 2 * FMA_XSLOT_BYTES);  // FMA
    float *red = (MODE == PATH_FMA)
                     ? reinterpret_cast<float *>(after + 2 * FMA_XSLOT_BYTES + FMA_PAIR_BYTES)
                     : reinterpret_cast<float *>(after);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = a.K / G;
    const int ntiles = (a.N + TILE_ROWS - 1) / TILE_ROWS;
    const int nrb = (ntiles + RB - 1) / RB;
    const int U = nrb * a.ks;
    const int xb = (a.xt == Q4_F32) ? 4 : 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], W);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == W) {
        if (lane == 0) {
            int gstep = 0, ui = 0, xissued = 0;
            bool ok = true;
            if (!a.debug_no_copy) {
                for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++ui) {
                    const UnitInfo un = unit_info(a, u, ntiles, NG);
                    if (MODE == PATH_FMA) {
                        const int xs = ui & 1;
                        if (ui >= 2 && !mbar_wait_bounded(&xempty[xs], ((ui >> 1) - 1) & 1,
                                                          abort_flag, a.wait_ns, a.err)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bytes =
                            static_cast<uint32_t>(un.g_end - un.g_begin) * G * xb;
                        mbar_arrive_expect_tx(&xfull[xs], bytes);
                        bulk_g2s(xslot + xs * FMA_XSLOT_BYTES,
                                 static_cast<const uint8_t *>(a.x) +
                                     static_cast<int64_t>(un.g_begin) * G * xb,
                                 bytes, &xfull[xs]);
                        ++xissued;
                    }
                    for (int ps = 0; ps < un.nsteps; ++ps, ++gstep) {
                        const int slot = gstep % NSTAGE;
                        if (gstep >= NSTAGE &&
                            !mbar_wait_bounded(&empty[slot], ((gstep / NSTAGE) - 1) & 1,
                                               abort_flag, a.wait_ns, a.err)) {
                            ok = false;
                            break;
                        }
                        const int g0 = un.g_begin + ps * W;
                        const int ng = min(W, un.g_end - g0);
                        const uint32_t row_bytes = static_cast<uint32_t>(ng) * TILE_BYTES;
                        mbar_arrive_expect_tx(&full[slot], row_bytes * un.nrt);
                        for (int r = 0; r < un.nrt; ++r) {
                            const uint8_t *src =
                                a.qw + (static_cast<int64_t>(un.rt0 + r) * NG + g0) * TILE_BYTES;
                            bulk_g2s(ring + slot * STAGE_BYTES + r * W * TILE_BYTES, src,
                                     row_bytes, &full[slot]);
                        }
                    }
                }
            }
            // Every issued copy must land before the CTA may exit.
            for (int s = max(0, gstep - NSTAGE); s < gstep; ++s)
                mbar_wait_bounded(&full[s % NSTAGE], (s / NSTAGE) & 1, abort_flag, a.wait_ns,
                                  a.err, false);
            for (int i = max(0, xissued - 2); i < xissued; ++i)
                mbar_wait_bounded(&xfull[i & 1], (i >> 1) & 1, abort_flag, a.wait_ns, a.err,
                                  false);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int gq = lane >> 2, t = lane & 3;
    const int M = a.M;
    const int MS = (MODE == PATH_FMA) ? 1 : 16;
    const int Mo = (MODE == PATH_FMA) ? 1 : M;
    const int npad = ntiles * TILE_ROWS;
    int gstep = 0, ui = 0;
    bool ok = true;

    for (int u = blockIdx.x; u < U; u += gridDim.x, ++ui) {
        const UnitInfo un = unit_info(a, u, ntiles, NG);

        if (MODE == PATH_FMA) {
            // Activation pairs in the order the code fields are extracted (see
            // the word layout in q4.h): per word, (x1,x8) (x9,x1) (x8,x0)
            // (x0',x9) with xa = x[16j + 2t + a] and x0' from the next word of
            // the same 16-byte chunk; plus S = sum x and the two offset terms.
            const int xs = ui & 1;
            ok = mbar_wait_bounded(&xfull[xs], (ui >> 1) & 1, abort_flag, a.wait_ns, a.err);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            const uint8_t *xsrc = xslot + xs * FMA_XSLOT_BYTES;
            const int ngs = un.g_end - un.g_begin;
            // record (gl, tt, j): one word's 8 pair floats; 32 records per
            // group, so every warp-wide pass covers whole (gl, tt) octets
            for (int base = 0; base < ngs * 32; base += CONSUMERS) {
                const int rec = base + threadIdx.x;
                const bool live = rec < ngs * 32;
                const int gl = rec >> 5, tt = (rec >> 3) & 3, j = rec & 7;
                const int jn = (j & 4) | ((j + 1) & 3);
                const int kb = gl * G + 2 * tt;
                float x0 = 0.0f, x1 = 0.0f, x8 = 0.0f, x9 = 0.0f, x0n = 0.0f;
                if (live) {
                    x0 = smem_x_f32(xsrc, a.xt, kb + 16 * j);
                    x1 = smem_x_f32(xsrc, a.xt, kb + 16 * j + 1);
                    x8 = smem_x_f32(xsrc, a.xt, kb + 16 * j + 8);
                    x9 = smem_x_f32(xsrc, a.xt, kb + 16 * j + 9);
                    x0n = smem_x_f32(xsrc, a.xt, kb + 16 * jn);
                    float4 *dst = reinterpret_cast<float4 *>(pairs + (gl * 4 + tt) * PAIR_STRIDE + 8 * j);
                    dst[0] = make_float4(x1, x8, x9, x1);
                    dst[1] = make_float4(x8, x0, x0n, x9);
                }
                // sums over the 8 words of this (gl, tt): lanes 8i..8i+7 share it
                float slo = x0 + x1, shi = x8 + x9;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    slo += __shfl_xor_sync(0xffffffffu, slo, o);
                    shi += __shfl_xor_sync(0xffffffffu, shi, o);
                }
                if (live && j == 0)
                    reinterpret_cast<float4 *>(pairs + FMA_PAIR_FLOATS)[gl * 4 + tt] =
                        make_float4(slo + shi, 128.0f * slo + 2048.0f * shi,
                                    128.0f * shi + 2048.0f * slo, 0.0f);
            }
            named_barrier_sync(1, CONSUMERS);
            if (lane == 0) mbar_arrive(&xempty[xs]);
        }

        float yacc[RB][NT][4];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) yacc[r][n][e] = 0.0f;

        // MMA: B fragments of the warp's group for the current step, and the
        // next step's prefetched while the current one computes (bf16/f16
        // activations; the f32 hi/lo split loads at step start).
        constexpr bool PREFETCH = (MODE == PATH_MMA) && !XSPLIT;
        uint32_t bcur[NT][8][2], bnxt[PREFETCH ? NT : 1][8][2];
        uint32_t blo[XSPLIT ? NT : 1][8][2];
        auto load_b = [&](int gg, uint32_t (&bh)[NT][8][2], uint32_t (&bl)[XSPLIT ? NT : 1][8][2]) {
            const bool act = gg < un.g_end;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int m = 8 * n + gq;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t k = static_cast<int64_t>(gg) * G + 16 * j + 2 * t;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t vh = 0, vl = 0;
                        if (act && m < M) {
                            const int64_t idx = static_cast<int64_t>(m) * a.K + k + 8 * h;
                            if (XSPLIT) {
                                const float2 xv = __ldg(reinterpret_cast<const float2 *>(
                                    static_cast<const float *>(a.x) + idx));
                                vh = pack_bf16x2(xv.x, xv.y);
                                vl = pack_bf16x2(xv.x - bf16_lo_f32(vh), xv.y - bf16_hi_f32(vh));
                            } else {
                                vh = __ldg(reinterpret_cast<const unsigned int *>(
                                    static_cast<const uint16_t *>(a.x) + idx));
                            }
                        }
                        bh[n][j][h] = vh;
                        if (XSPLIT) bl[XSPLIT ? n : 0][j][h] = vl;
                    }
                }
            }
        };
        if (MODE == PATH_MMA) load_b(un.g_begin + warp, bcur, blo);

        for (int s = 0; s < un.nsteps; ++s, ++gstep) {
            const int slot = gstep % NSTAGE;
            const int g = un.g_begin + s * W + warp;
            const bool active = g < un.g_end;

            ok = mbar_wait_bounded(&full[slot], (gstep / NSTAGE) & 1, abort_flag, a.wait_ns, a.err);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            if (MODE == PATH_MMA && XSPLIT && s > 0) load_b(g, bcur, blo);
            if (PREFETCH && s + 1 < un.nsteps)
                load_b(g + W, reinterpret_cast<uint32_t (&)[NT][8][2]>(bnxt), blo);
            const uint8_t *stage = ring + slot * STAGE_BYTES + warp * TILE_BYTES;
            if (active && MODE == PATH_FMA) {
                const int gl = g - un.g_begin;
                const float4 *xpp =
                    reinterpret_cast<const float4 *>(pairs + (gl * 4 + t) * PAIR_STRIDE);
                float2 P[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 p = xpp[2 * j], q = xpp[2 * j + 1];
                    P[j][0] = make_float2(p.x, p.y);
                    P[j][1] = make_float2(p.z, p.w);
                    P[j][2] = make_float2(q.x, q.y);
                    P[j][3] = make_float2(q.z, q.w);
                }
                const float4 xsv = reinterpret_cast<const float4 *>(pairs + FMA_PAIR_FLOATS)[gl * 4 + t];
                // all RB tiles at once: RB independent accumulator chains
                uint32_t wv[RB][8];
                float2 sp[RB];
                uint32_t zp[RB];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const uint8_t *tile = stage + r * W * TILE_BYTES;
                    const bool live = r < un.nrt;
                    const uint4 c0 = live ? *reinterpret_cast<const uint4 *>(tile + 16 * lane)
                                          : make_uint4(0, 0, 0, 0);
                    const uint4 c1 = live ? *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane)
                                          : make_uint4(0, 0, 0, 0);
                    sp[r] = live ? *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq)
                                 : make_float2(0.0f, 0.0f);
                    zp[r] = live ? *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq) : 0u;
                    wv[r][0] = c0.x; wv[r][1] = c0.y; wv[r][2] = c0.z; wv[r][3] = c0.w;
                    wv[r][4] = c1.x; wv[r][5] = c1.y; wv[r][6] = c1.z; wv[r][7] = c1.w;
                }
                float2 accG[RB], accG8[RB];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    accG[r] = make_float2(0.0f, 0.0f);
                    accG8[r] = make_float2(0.0f, 0.0f);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        const uint32_t wj = wv[r][j], wn = wv[r][(j & 4) | ((j + 1) & 3)];
                        accG[r] = __ffma2_rn(code_pair(wj), P[j][0], accG[r]);
                        accG8[r] = __ffma2_rn(code_pair(wj >> 8), P[j][1], accG8[r]);
                        accG8[r] = __ffma2_rn(code_pair(wj << 8), P[j][2], accG8[r]);
                        accG[r] = __ffma2_rn(code_pair(__funnelshift_r(wj, wn, 16)), P[j][3], accG[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float zg = static_cast<float>(zp[r] & 0xFFu);
                    const float zg8 = static_cast<float>(zp[r] >> 8);
                    const float ig =
                        fmaf(128.0f, accG[r].x, fmaf(2048.0f, accG[r].y, -fmaf(zg, xsv.x, xsv.y)));
                    const float ig8 =
                        fmaf(128.0f, accG8[r].x, fmaf(2048.0f, accG8[r].y, -fmaf(zg8, xsv.x, xsv.z)));
                    yacc[r][0][0] = fmaf(sp[r].x, ig, yacc[r][0][0]);
                    yacc[r][0][2] = fmaf(sp[r].y, ig8, yacc[r][0][2]);
                }
            } else if (active && MODE == PATH_MMA) {
                const uint32_t MAG = ABT == 0 ? 0x43004300u : 0x64006400u;
                const uint32_t ONES = ABT == 0 ? 0x3F803F80u : 0x3C003C00u;
                const float OFF = ABT == 0 ? 128.0f : 1024.0f;
                // TI tiles at a time: TI * NT independent accumulator chains,
                // plus NT chains for the activation sums
                constexpr int TI = (NT == 1) ? 4 : 2;
                float S[NT][4];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) S[n][e] = 0.0f;
#pragma unroll
                for (int r0 = 0; r0 < RB; r0 += TI) {
                    uint32_t wv[TI][8];
                    float2 sp[TI];
                    uint32_t zp[TI];
#pragma unroll
                    for (int i = 0; i < TI; ++i) {
                        const uint8_t *tile = stage + (r0 + i) * W * TILE_BYTES;
                        const bool live = r0 + i < un.nrt;
                        const uint4 c0 = live ? *reinterpret_cast<const uint4 *>(tile + 16 * lane)
                                              : make_uint4(0, 0, 0, 0);
                        const uint4 c1 = live ? *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane)
                                              : make_uint4(0, 0, 0, 0);
                        sp[i] = live ? *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq)
                                     : make_float2(0.0f, 0.0f);
                        zp[i] = live ? *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq) : 0u;
                        wv[i][0] = c0.x; wv[i][1] = c0.y; wv[i][2] = c0.z; wv[i][3] = c0.w;
                        wv[i][4] = c1.x; wv[i][5] = c1.y; wv[i][6] = c1.z; wv[i][7] = c1.w;
                    }
                    float d[TI][NT][4];
#pragma unroll
                    for (int i = 0; i < TI; ++i)
#pragma unroll
                        for (int n = 0; n < NT; ++n)
#pragma unroll
                            for (int e = 0; e < 4; ++e) d[i][n][e] = 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (r0 == 0) {
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                mma_ab<ABT>(S[n], ONES, ONES, ONES, ONES, bcur[n][j][0], bcur[n][j][1]);
                                if (XSPLIT)
                                    mma_ab<ABT>(S[n], ONES, ONES, ONES, ONES, blo[XSPLIT ? n : 0][j][0],
                                                blo[XSPLIT ? n : 0][j][1]);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < TI; ++i) {
                            const uint32_t w = wv[i][j];
                            const uint32_t a0 = lop3_and_or(w, 0x000F000Fu, MAG);
                            const uint32_t a1 = lop3_and_or(w >> 4, 0x000F000Fu, MAG);
                            const uint32_t a3 = lop3_and_or(w >> 8, 0x000F000Fu, MAG);
                            const uint32_t a2 = lop3_and_or(w >> 12, 0x000F000Fu, MAG);
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                mma_ab<ABT>(d[i][n], a0, a1, a2, a3, bcur[n][j][0], bcur[n][j][1]);
                                if (XSPLIT)
                                    mma_ab<ABT>(d[i][n], a0, a1, a2, a3, blo[XSPLIT ? n : 0][j][0],
                                                blo[XSPLIT ? n : 0][j][1]);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < TI; ++i) {
                        const float zg = OFF + static_cast<float>(zp[i] & 0xFFu);
                        const float zg8 = OFF + static_cast<float>(zp[i] >> 8);
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            float *ya = yacc[r0 + i][n];
                            ya[0] = fmaf(sp[i].x, fmaf(-zg, S[n][0], d[i][n][0]), ya[0]);
                            ya[1] = fmaf(sp[i].x, fmaf(-zg, S[n][1], d[i][n][1]), ya[1]);
                            ya[2] = fmaf(sp[i].y, fmaf(-zg8, S[n][0], d[i][n][2]), ya[2]);
                            ya[3] = fmaf(sp[i].y, fmaf(-zg8, S[n][1], d[i][n][3]), ya[3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (PREFETCH) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        bcur[n][j][0] = bnxt[PREFETCH ? n : 0][j][0];
                        bcur[n][j][1] = bnxt[PREFETCH ? n : 0][j][1];
                    }
            }
        }
        if (!ok) break;

        // ------------------------------------------- reduction and output
        if (MODE == PATH_FMA) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float v = yacc[r][0][0], v8 = yacc[r][0][2];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v8 += __shfl_xor_sync(0xffffffffu, v8, 1);
                v8 += __shfl_xor_sync(0xffffffffu, v8, 2);
                if (t == 0) {
                    red[warp * RB * 16 + r * 16 + gq] = v;
                    red[warp * RB * 16 + r * 16 + gq + 8] = v8;
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
        named_barrier_sync(1, CONSUMERS);

        const int nout = un.nrt * 16 * Mo;
        const int row0 = un.rt0 * TILE_ROWS;
        for (int i = threadIdx.x; i < nout; i += CONSUMERS) {
            const int row = i / Mo, m = i % Mo;
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < W; ++w) v += red[(w * RB * 16 + row) * MS + m];
            if (a.ks == 1) {
                if (row0 + row < a.N)
                    store_y(a.y, a.yt, static_cast<int64_t>(m) * a.N + row0 + row, v);
            } else {
                a.partial[(static_cast<int64_t>(un.ks) * M + m) * npad + row0 + row] = v;
            }
        }
        if (a.ks > 1) {
            // Split over K: the last unit of this row block sums the slices in
            // order.  One thread publishes the CTA's partials (the barrier
            // orders the other threads' stores before its release fence) and
            // acquires the others' before the barrier that releases the reads.
            named_barrier_sync(1, CONSUMERS);
            if (threadIdx.x == 0) {
                __threadfence();
                const unsigned int prev = atomicAdd(&a.count[un.rb], 1u);
                __threadfence();
                *last_flag = (prev == static_cast<unsigned int>(a.ks - 1));
            }
            named_barrier_sync(1, CONSUMERS);
            if (*last_flag) {
                for (int i = threadIdx.x; i < nout; i += CONSUMERS) {
                    const int row = i / Mo, m = i % Mo;
                    if (row0 + row >= a.N) continue;
                    float v = 0.0f;
                    for (int s2 = 0; s2 < a.ks; ++s2)
                        v += __ldcg(&a.partial[(static_cast<int64_t>(s2) * M + m) * npad + row0 + row]);
                    store_y(a.y, a.yt, static_cast<int64_t>(m) * a.N + row0 + row, v);
                }
                if (threadIdx.x == 0) a.count[un.rb] = 0u;  // ready for the next call
            }
        }
        // red, pairs and last_flag are reused by the next unit
        named_barrier_sync(1, CONSUMERS);
    }
}

// -------------------------------------------------------------------- host
template <int MODE, int NT, int ABT, bool XSPLIT>
struct Kern {
    static cudaError_t configure(int dev, int *blocks_per_sm)
    {
        static int cached[64] = {};
        if (dev >= 0 && dev < 64 && cached[dev] > 0) {
            *blocks_per_sm = cached[dev];
            return cudaSuccess;
        }
        auto kern = k_gemv<MODE, NT, ABT, XSPLIT>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes(MODE));
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, THREADS, smem_bytes(MODE));
        if (e != cudaSuccess) return e;
        if (n < 1) n = 1;
        if (dev >= 0 && dev < 64) cached[dev] = n;
        *blocks_per_sm = n;
        return cudaSuccess;
    }
    static cudaError_t launch(int grid, const GemvArgs &a, cudaStream_t s)
    {
        k_gemv<MODE, NT, ABT, XSPLIT><<<grid, THREADS, smem_bytes(MODE), s>>>(a);
        return cudaGetLastError();
    }
};

template <typename F>
static cudaError_t dispatch(int path, int M, q4_dtype xt, F &&f)
{
    if (path == PATH_FMA) return f(Kern<PATH_FMA, 1, 0, false>{});
    const bool two = M > 8;
    if (xt == Q4_F16) return two ? f(Kern<PATH_MMA, 2, 1, false>{}) : f(Kern<PATH_MMA, 1, 1, false>{});
    if (xt == Q4_BF16) return two ? f(Kern<PATH_MMA, 2, 0, false>{}) : f(Kern<PATH_MMA, 1, 0, false>{});
    return two ? f(Kern<PATH_MMA, 2, 0, true>{}) : f(Kern<PATH_MMA, 1, 0, true>{});
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
    int dev = 0, per_sm = 1;
    cudaGetDevice(&dev);
    dispatch(path, M, xt, [&](auto k) { return decltype(k)::configure(dev, &per_sm); });
    const long slots = static_cast<long>(sm_count) * per_sm;
    const int gs_max = (path == PATH_FMA) ? GS_MAX_FMA : GS_MAX_MMA;
    // Pick the K slice: units per CTA slot rounded up (the static round-robin
    // tail) times the work per unit (steps of W groups plus about one step of
    // per-unit overhead), plus the split-K partial traffic in step units.
    double best = -1.0;
    int best_gs = NG < gs_max ? NG : gs_max;
    for (int gs = (NG < gs_max ? NG : gs_max); gs >= 1; --gs) {
        const int ks = (NG + gs - 1) / gs;
        if ((ks - 1) * gs >= NG) continue;
        const long units = static_cast<long>(p.nrb) * ks;
        const long per_cta = (units + slots - 1) / slots;
        const double steps = (gs + W - 1) / W + 1.0 + (ks > 1 ? 0.5 : 0.0);
        const double partial = ks > 1 ? 8.0 * ks * M / (0.539 * K) * (NG / 4.0) : 0.0;
        const double cost = static_cast<double>(per_cta) * steps * slots / p.nrb + partial;
        if (best < 0 || cost < best - 1e-9) {
            best = cost;
            best_gs = gs;
        }
    }
    p.gs = best_gs;
    p.ks = (NG + best_gs - 1) / best_gs;
    p.grid = static_cast<int>(std::min<long>(static_cast<long>(p.nrb) * p.ks, slots));
    p.workspace = p.ks > 1 ? counters_bytes(p.nrb) + static_cast<size_t>(p.ks) * M * ntiles *
                                                         TILE_ROWS * sizeof(float)
                           : 0;
    return p;
}

cudaError_t gemv_launch(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    return dispatch(p.path, a.M, a.xt, [&](auto k) { return decltype(k)::launch(p.grid, a, s); });
}

}  // namespace q4
