// gemm_tc.cu -- W4A16 GEMM on the sm_103a tcgen05 tensor cores, exact per group.
//
// Y[M][N] = X[M][K] * W_hat[N][K]^T with W_hat = (q - zero) * scale per group
// of 128 along K (page "Weight quantization", "How it works"), computed the
// way that page factors the product, one multiply per group: for every group
// g the tensor cores form
//     D_g[n][m] = sum_{k in g} (q[n][k] - zero[n][g]) * x[m][k]
// from the small integers q - zero (exact in bf16 or f16, the activations'
// type) with f32 accumulation in tensor memory, and
//     Y^T[n][m] += scale[n][g] * D_g[n][m]
// is added up in f32 registers.  No weight is ever rounded to 16 bits, so the
// result differs from the exact product by f32 rounding only.  The packed
// codes are unpacked on chip and the floating-point weights never reach HBM
// (page "LLM Quantization Architecture in Depth", "Kernels and memory
// layout").
//
// One persistent CTA per SM, 20 warps with fixed roles (a warp reaches the
// tensor-memory lanes of quadrant warp % 4 only, and runs on SM partition
// warp % 4):
//   warp 0      activation producer: X tiles by 2-D tensor TMA (128-byte
//               swizzle, K-major), one stage per group;
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma;
//   warp 19     weight producer: the group's 8 packed tiles (16 rows each)
//               by 1-D bulk copies into a ring of code stages (on partition
//               3, which has no other producer: the builders of the
//               partition that also runs a producer fall behind the others,
//               and the MMAs wait for the slowest builder; warp 2 idles);
//   warps 3-10  operand builders, two per tensor-memory lane quadrant (one
//               per half of the group's k): each thread owns one weight row,
//               turns its 64 codes into 32 packed (q - zero) pairs with a
//               shift, one LOP3 and one packed FMA per pair, and stores them
//               with tcgen05.st as the MMA's A operand (tensor memory, not
//               shared memory: shared memory carries only the activations and
//               the packed codes);
//   warps 11-18 rescale and epilogue, two per quadrant (each half of the
//               tile's token columns): per group each thread loads its row's
//               D_g columns (tcgen05.ld), releases the buffer and adds
//               scale * D_g into its f32 accumulators; at the end of a tile
//               it stores the row (or a partial sum, below).
// Tensor memory (512 columns): D_g double-buffered in columns [0, 256) and
// the A stages of one group each at 256 + 64 s.  With at most 64 tokens a
// group's 8 MMAs alternate between two accumulators (its two k halves,
// summed by the rescale): an MMA of fewer than 128 columns takes about 51
// cycles however small, so a single dependent chain of 8 would leave the
// tensor core idle.
// A CTA tile is 128 weight rows x BT tokens, BT the smallest of 16, 32, 64,
// 128 that covers M (128 beyond): 128 x BT x 16 MMAs, A from tensor memory,
// B = the activation rows from shared memory.
// Per group the MMA thread waits for two barriers (its D buffer free, A
// built and the activations landed -- one operand builder waits for the
// latter before it arrives) and commits once: that one commit frees the
// activation and A stage and hands D_g to the rescale warps.
//
// Work: when there are many tiles every CTA takes whole tiles in turn; when
// there are few (a few dozen tokens), the tiles' groups form one sequence of
// items cut into equal contiguous ranges, one per CTA, and a tile whose
// groups are spread over several CTAs is finished by the last of them to
// arrive, which adds the f32 partial sums of all contributors in CTA order
// (results do not depend on timing) and clears them for the next call.
//
// Every barrier wait is bounded; on expiry the CTA raises the device error
// word, every role stops, the copies and tensor-core operations in flight are
// waited for, tensor memory is freed and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace q4 {
namespace gm {

constexpr int BN = 128;                    // weight rows per tile
constexpr int RT = BN / TILE_ROWS;         // 8 packed tiles per group
static_assert(RT == LB_TILES, "a tile's row tiles form one block of the weight layout");
constexpr int C_STAGE = RT * TILE_BYTES;   // 8832 bytes of codes per group (compact: 8576 used)
#ifndef GEMM_WPROD
#define GEMM_WPROD 19
#endif
// The weight producer has a warp of its own on SM partition 3, the one
// partition without a producer or the MMA thread (a warp reaches the
// tensor-memory lanes of its partition only, so every partition already
// runs two operand builders and two rescale warps); warp 2 idles.
constexpr int WPROD = GEMM_WPROD;
constexpr int THREADS = (WPROD == 19 ? 20 : 19) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL = 256;            // first tensor-memory column of the A stages
constexpr int NS = 4;                      // activation / A stages
constexpr int NSC = 8;                     // scale hand-off slots
constexpr int BAND = 8;                    // token tiles per raster band

template <int BT>
struct Plan {
    static constexpr int NC = BT >= 128 ? 6 : 8;  // code stages
    static constexpr int X_HALF = BT * 64 * 2;    // one 64-k half of a group's activations
    static constexpr int X_ST = 2 * X_HALF;
    static constexpr int OFF_X = 0;
    static constexpr int OFF_C = NS * X_ST;
    static constexpr int OFF_S = ((OFF_C + NC * C_STAGE + 15) / 16) * 16;  // scale slots
    static constexpr int OFF_BAR = OFF_S + NSC * BN * 4;
    static constexpr int NBAR = 3 * NS + 2 * NC + NSC + 3;
    static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
    static_assert(X_HALF % 1024 == 0, "swizzled halves start on 1024-byte boundaries");
    static_assert(SMEM_ALLOC <= 227 * 1024, "one CTA per SM");
};

// ----------------------------------------------------------------- PTX
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (tcgen05 descriptor format, version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;    // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;  // stride byte offset: next 8-row group
    d |= static_cast<uint64_t>(1) << 46;           // descriptor version
    d |= static_cast<uint64_t>(2) << 61;           // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: f32 accumulate, A/B bf16 (ab = 1) or
// f16 (ab = 0), both K-major, M = 128, N = n (a multiple of 16, 16..256).
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab, uint32_t n)
{
    return (1u << 4) | (ab << 7) | (ab << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

// D (tensor memory) [+]= A (tensor memory) * B (shared memory descriptor).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

#define Q4_R8(a, o) "r"(a[o + 0]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), "r"(a[o + 4]), \
    "r"(a[o + 5]), "r"(a[o + 6]), "r"(a[o + 7])
#define Q4_W8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
    "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])

// 32 consecutive 32-bit columns of this warp's 32 lanes <- v (thread i: lane i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        Q4_R8(v, 0), Q4_R8(v, 8), Q4_R8(v, 16), Q4_R8(v, 24)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// v <- consecutive columns of this warp's lanes; complete at tmem_wait_ld.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : Q4_W8(v, 0)
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16x(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15}, [%16];"
        : Q4_W8(v, 0), Q4_W8(v, 8)
        : "r"(taddr)
        : "memory");
}
#undef Q4_R8
#undef Q4_W8

// C consecutive 32-bit columns (C = 8 or 16) of this warp's lanes.
template <int C>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[C])
{
    if constexpr (C == 8)
        tmem_ld8(taddr, v);
    else
        tmem_ld16x(taddr, v);
}

struct Args {
    const uint8_t *qw;
    void *y;
    q4_dtype yt;
    int M, N, K;
    int mt, nt;            // tiles along M (bt tokens) and N (128 rows)
    int split;             // 1: contiguous item ranges, partial sums through the workspace
    int maxc;              // most CTAs sharing one tile
    unsigned int *count;   // [tiles] arrival counters (split)
    float *partial;        // [tiles][maxc][128 rows][bt] partial sums (split)
    int64_t count_len;     // extents of the two, for the store checks of debug builds
    int64_t partial_len;
    uint64_t wait_ns;
    unsigned int *err;
    int debug_no_copy;     // the weight producer copies nothing (bounded-wait self-test)
};

// Tile t of the raster: bands of BAND token tiles; inside a band the token
// tile runs fastest, so the CTAs working at the same time share few weight
// tiles and few activation tiles.
__device__ __forceinline__ void tile_coords(int t, int mt, int nt, int &mb, int &nb)
{
    const int band = t / (BAND * nt);
    const int bm = min(BAND, mt - band * BAND);
    const int r = t - band * BAND * nt;
    mb = band * BAND + r % bm;
    nb = r / bm;
}

// The CTA's next unit of work: a tile and its group range [g0, g1).
struct Cursor {
    int64_t pos, end;
};
__device__ __forceinline__ bool next_unit(const Args &a, int NG, Cursor &c, int &tile, int &g0,
                                          int &g1)
{
    if (c.pos >= c.end) return false;
    if (a.split) {
        tile = static_cast<int>(c.pos / NG);
        g0 = static_cast<int>(c.pos % NG);
        const int64_t left = c.end - c.pos;
        g1 = static_cast<int>(left < NG - g0 ? g0 + left : NG);
        c.pos += g1 - g0;
    } else {
        tile = static_cast<int>(c.pos);
        g0 = 0;
        g1 = NG;
        c.pos += gridDim.x;
    }
    return true;
}

// CTA owning item i of T items split over G CTAs (contiguous equal ranges).
__device__ __forceinline__ int64_t owner_of(int64_t i, int64_t T, int64_t G) { return ((i + 1) * G - 1) / T; }

__device__ __forceinline__ void store_out(void *y, q4_dtype yt, int64_t idx, float v)
{
    if (yt == Q4_F32)
        static_cast<float *>(y)[idx] = v;
    else if (yt == Q4_BF16)
        static_cast<__nv_bfloat16 *>(y)[idx] = __float2bfloat16_rn(v);
    else
        static_cast<__half *>(y)[idx] = __float2half_rn(v);
}

// The epilogue's global stores, each checked against its buffer in debug
// builds (a store outside it is recorded and skipped).
__device__ __forceinline__ void put_out(const Args &a, int64_t idx, float v)
{
    if (store_ok(idx, static_cast<int64_t>(a.M) * a.N, a.err)) store_out(a.y, a.yt, idx, v);
}
__device__ __forceinline__ void put_part4(const Args &a, float4 *p, float4 v)
{
    if (store_ok(reinterpret_cast<float *>(p) - a.partial + 3, a.partial_len, a.err)) *p = v;
}
__device__ __forceinline__ bool count_ok(const Args &a, int tile)
{
    return store_ok(tile, a.count_len, a.err);
}

// F16: activations (and the A operand) are f16, else bf16.  BT: tokens per
// tile.  CMP: compact tiles (binary16 scale pairs, zero nibbles, 1072 bytes).
template <bool F16, int BT, bool CMP>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmx, const Args a)
{
    using P = Plan<BT>;
    constexpr int NC = P::NC, X_HALF = P::X_HALF, X_ST = P::X_ST;
    constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    constexpr int NCOL = BT >= 128 ? 64 : BT / 2;  // token columns per rescale thread
    constexpr int CH = NCOL < 16 ? NCOL : 16;        // columns per tensor-memory load
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem + P::OFF_X;
    uint8_t *sC = smem + P::OFF_C;
    float *sScl = reinterpret_cast<float *>(smem + P::OFF_S);  // [NSC][128 rows]
    // xfull: activations landed; afull: A built (8 builders); mdone: the
    // group's MMAs completed (frees the stage, hands D_g over); cfull/cempty:
    // code stages; sfull: scales handed over; dempty: D buffer read.
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P::OFF_BAR);
    uint64_t *xfull = bar, *afull = xfull + NS, *mdone = afull + NS;
    uint64_t *cfull = mdone + NS, *cempty = cfull + NC;
    uint64_t *sfull = cempty + NC;
    uint64_t *dempty = sfull + NSC, *drain = dempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile unsigned int *bcast = reinterpret_cast<volatile unsigned int *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = a.K / G;
    const int ntiles_rows = (a.N + TILE_ROWS - 1) / TILE_ROWS;
    const int64_t T = static_cast<int64_t>(a.mt) * a.nt;
    const int64_t items = T * NG;
    Cursor cur0;
    if (a.split) {
        cur0.pos = blockIdx.x * items / gridDim.x;
        cur0.end = (blockIdx.x + 1) * items / gridDim.x;
    } else {
        cur0.pos = blockIdx.x;
        cur0.end = T;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&afull[i], 8);
            mbar_init(&mdone[i], 1);
        }
        for (int i = 0; i < NC; ++i) {
            mbar_init(&cfull[i], 1);
            mbar_init(&cempty[i], 8);
        }
        for (int i = 0; i < NSC; ++i) mbar_init(&sfull[i], 4);
        for (int i = 0; i < 2; ++i) mbar_init(&dempty[i], 8);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------- activation producer
        if (lane == 0) {
            Cursor cur = cur0;
            int tile, g0, g1, i = 0;
            bool ok = true;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                int mb, nb;
                tile_coords(tile, a.mt, a.nt, mb, nb);
                for (int g = g0; g < g1; ++g) {
                    const int s = i % NS;
                    if (i >= NS && !mbar_wait_bounded(&mdone[s], ((i / NS) - 1) & 1, abort_flag,
                                                      a.wait_ns, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&xfull[s], static_cast<uint32_t>(X_ST));
                    uint8_t *dst = sX + s * X_ST;
                    tma_load_2d(dst, &tmx, g * G, mb * BT, &xfull[s]);
                    tma_load_2d(dst + X_HALF, &tmx, g * G + 64, mb * BT, &xfull[s]);
                    ++i;
                }
            }
            // every issued copy lands before the CTA may exit
            for (int j = max(0, i - NS); j < i; ++j)
                mbar_wait_bounded(&xfull[j % NS], (j / NS) & 1, abort_flag, a.wait_ns, a.err, false);
        }
    } else if (warp == WPROD) {
        // ----------------------------------------------------- weight producer
        if (lane == 0 && !a.debug_no_copy) {
            Cursor cur = cur0;
            int tile, g0, g1, i = 0;
            bool ok = true;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                int mb, nb;
                tile_coords(tile, a.mt, a.nt, mb, nb);
                const int rt0 = nb * RT, nrt = min(RT, ntiles_rows - rt0);
                for (int g = g0; g < g1; ++g) {
                    const int c = i % NC;
                    if (i >= NC && !mbar_wait_bounded(&cempty[c], ((i / NC) - 1) & 1, abort_flag,
                                                      a.wait_ns, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&cfull[c], static_cast<uint32_t>(nrt) * TBY);
                    // the tile's 8 row tiles lie in one block of the weight
                    // layout: group g of each, ng tiles apart
                    const int64_t t0 = tile_index(rt0, g, ntiles_rows, NG);
                    const int ng = min(LB_GROUPS, NG - (g / LB_GROUPS) * LB_GROUPS);
                    for (int r = 0; r < nrt; ++r)
                        bulk_g2s(sC + c * C_STAGE + r * TBY, a.qw + (t0 + r * ng) * TBY, TBY, &cfull[c]);
                    ++i;
                }
            }
            for (int j = max(0, i - NC); j < i; ++j)
                mbar_wait_bounded(&cfull[j % NC], (j / NC) & 1, abort_flag, a.wait_ns, a.err, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(F16 ? 0u : 1u, static_cast<uint32_t>(BT));
            Cursor cur = cur0;
            int tile, g0, g1, i = 0;
            bool ok = true, issued = false;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                for (int g = g0; g < g1; ++g, ++i) {
                    const int s = i % NS, b = i & 1;
                    // the MMA thread polls (reacts at once; it has nothing else to do)
                    if ((i >= 2 && !mbar_wait_bounded(&dempty[b], ((i >> 1) - 1) & 1, abort_flag,
                                                      a.wait_ns, a.err, true, true)) ||
                        !mbar_wait_bounded(&afull[s], (i / NS) & 1, abort_flag, a.wait_ns, a.err,
                                           true, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // one descriptor per stage; a k step's operand lies a
                    // constant number of 16-byte units further on
                    const uint64_t xd = sw128_desc(smem_u32(sX + s * X_ST));
                    const uint32_t at = tmem + A_COL + static_cast<uint32_t>(s) * 64u;
                    if constexpr (BT <= 64) {
                        // two accumulators (k halves 0-63 and 64-127), interleaved
                        const uint32_t d0 = tmem + static_cast<uint32_t>(b) * 128u;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            mma_ts(d0, at + 8u * k, xd + (32 * k) / 16, idesc, k > 0 ? 1u : 0u);
                            mma_ts(d0 + 64u, at + 32u + 8u * k, xd + (X_HALF + 32 * k) / 16, idesc,
                                   k > 0 ? 1u : 0u);
                        }
                    } else {
                        const uint32_t d = tmem + static_cast<uint32_t>(b) * 128u;
#pragma unroll
                        for (int k16 = 0; k16 < 8; ++k16)
                            mma_ts(d, at + 8u * k16, xd + ((k16 >> 2) * X_HALF + 32 * (k16 & 3)) / 16,
                                   idesc, k16 > 0 ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit(&mdone[s]);
                }
            }
            if (issued) {
                // all issued MMAs complete before tensor memory is freed
                mma_commit(drain);
                mbar_wait_bounded(drain, 0, abort_flag, a.wait_ns, a.err, false);
            }
        }
    } else if (warp >= 3 && warp < 11) {
        // ------------------------------------------------ A operand builders
        // Thread = weight row R of the tile (tensor-memory lane R); builder
        // warp w (w % 4 = q) builds k half (w - 3) / 4 of lane quadrant q.  The row's codes sit
        // in lanes 4 (R % 8) + t of its packed tile (t = 0..3), in the nibble
        // fields of row R % 16 (tiled layout, include/q4.h): word i of chunk
        // h of lane 4 (R % 8) + t holds k = 16 (4h + i) + 2t + {0, 1} and
        // + {8, 9}, i.e. the packed pairs 32h + 8i + t and 32h + 8i + t + 4
        // of the group's 64.
        const int q = warp & 3, kh = (warp - 3) >> 2;
        const int R = 32 * q + lane, d = R >> 4, rr = R & 15;
        const int lg = 4 * (rr & 7);
        const uint32_t sA = (rr & 8) ? 4u : 0u, sB = (rr & 8) ? 8u : 12u;
        const uint32_t MAG = F16 ? 0x64006400u : 0x43004300u;
        const float OFF = F16 ? 1024.0f : 128.0f;
        const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q) << 16) + A_COL + 32u * kh;
        Cursor cur = cur0;
        int tile, g0, g1, i = 0;
        bool ok = true;
        while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
            int mb, nb;
            tile_coords(tile, a.mt, a.nt, mb, nb);
            const int nrt = min(RT, ntiles_rows - nb * RT);
            const bool live = d < nrt;
            for (int g = g0; g < g1; ++g) {
                const int c = i % NC, s = i % NS, sl = i % NSC;
                // A stage s and scale slot sl are free once the MMAs of group
                // i - NS completed: those waited for the rescale of group
                // i - NS - 2 to release its D buffer, after it had read its
                // scale slot, and slot sl's previous user, group i - NSC, is
                // older still.
                ok = mbar_wait_bounded(&cfull[c], (i / NC) & 1, abort_flag, a.wait_ns, a.err);
                if (ok && i >= NS)
                    ok = mbar_wait_bounded(&mdone[s], ((i / NS) - 1) & 1, abort_flag, a.wait_ns,
                                           a.err);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const uint8_t *ct = sC + c * C_STAGE + d * TBY;
                uint32_t mz = 0;
                if (live) {
                    int z;
                    float sc;
                    if (CMP) {
                        sc = __half2float(*reinterpret_cast<const __half *>(
                            ct + SCALE_OFF + 4 * (rr & 7) + 2 * (rr >> 3)));
                        z = (ct[CMP_ZERO_OFF + (rr & 7)] >> (4 * (rr >> 3))) & 15;
                    } else {
                        sc = *reinterpret_cast<const float *>(ct + SCALE_OFF + 8 * (rr & 7) +
                                                             4 * (rr >> 3));
                        z = ct[ZERO_OFF + 2 * (rr & 7) + (rr >> 3)];
                    }
                    if (kh == 0) sScl[sl * BN + R] = sc;
                    const float nz = -(OFF + static_cast<float>(z));  // exact in 16 bits
                    if (F16) {
                        const __half2 h = __floats2half2_rn(nz, nz);
                        mz = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(nz, nz);
                        mz = *reinterpret_cast<const uint32_t *>(&h);
                    }
                } else if (kh == 0) {
                    sScl[sl * BN + R] = 0.0f;
                }
                uint32_t v[32];
                if (live) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint4 w4 = *reinterpret_cast<const uint4 *>(ct + kh * 512 + 16 * (lg + t));
                        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int i4 = 0; i4 < 4; ++i4) {
                            v[8 * i4 + t] = sub_pair<F16>(lop3_and_or(ws[i4] >> sA, 0x000F000Fu, MAG), mz);
                            v[8 * i4 + t + 4] = sub_pair<F16>(lop3_and_or(ws[i4] >> sB, 0x000F000Fu, MAG), mz);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;  // rows past the matrix
                }
                tmem_st32(tlane + static_cast<uint32_t>(s) * 64u, v);
                tmem_wait_st();
                tc_fence_before();
                // one builder also waits for the stage's activations, so that
                // A built = everything the MMAs of group i read is in place
                bool landed = true;
                if (warp == 3)
                    landed = mbar_wait_bounded(&xfull[s], (i / NS) & 1, abort_flag, a.wait_ns, a.err);
                __syncwarp();
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive(&afull[s]);
                    mbar_arrive(&cempty[c]);
                    if (kh == 0) mbar_arrive(&sfull[sl]);
                }
                ++i;
            }
        }
    } else if (warp >= 11 && warp < 19) {
        // ------------------------------------------------ rescale + epilogue
        const int w = warp - 11, q = warp & 3, ch = w >> 2;
        const int R = 32 * q + lane;
        const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(NCOL * ch);
        Cursor cur = cur0;
        int tile, g0, g1, i = 0;
        bool ok = true;
        while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
            int mb, nb;
            tile_coords(tile, a.mt, a.nt, mb, nb);
            const int n = nb * BN + R;
            float Y[NCOL];
#pragma unroll
            for (int j = 0; j < NCOL; ++j) Y[j] = 0.0f;
            for (int g = g0; g < g1; ++g) {
                const int s = i % NS, b = i & 1, sl = i % NSC;
                ok = mbar_wait_bounded(&mdone[s], (i / NS) & 1, abort_flag, a.wait_ns, a.err) &&
                     mbar_wait_bounded(&sfull[sl], (i / NSC) & 1, abort_flag, a.wait_ns, a.err);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float sc = sScl[sl * BN + R];
                const uint32_t db = tlane + static_cast<uint32_t>(b) * 128u;
                // this thread's NCOL columns, CH at a time (with at most 64
                // tokens also the second k half's accumulator, 64 columns
                // on); the buffer is released once the last chunk is loaded
#pragma unroll
                for (int c0 = 0; c0 < NCOL; c0 += CH) {
                    uint32_t v[CH], u[CH];
                    tmem_ld<CH>(db + c0, v);
                    if constexpr (BT <= 64) tmem_ld<CH>(db + 64u + c0, u);
                    tmem_wait_ld();
                    if (c0 + CH == NCOL) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&dempty[b]);
                    }
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const float dv = BT <= 64 ? __uint_as_float(v[j]) + __uint_as_float(u[j])
                                                  : __uint_as_float(v[j]);
                        Y[c0 + j] = fmaf(sc, dv, Y[c0 + j]);
                    }
                }
                ++i;
            }

            // ---------------------------------------------------- tile output
            const int64_t first = static_cast<int64_t>(tile) * NG;
            int c_first = blockIdx.x, nc = 1;
            if (a.split) {
                c_first = static_cast<int>(owner_of(first, items, gridDim.x));
                nc = static_cast<int>(owner_of(first + NG - 1, items, gridDim.x)) - c_first + 1;
                // every rescale warp decides together whether to go on
                if (named_barrier_or(1, 256, !ok)) {
                    ok = false;
                    break;
                }
            } else if (!ok) {
                break;
            }
            const int m0 = mb * BT + NCOL * ch;
            if (nc == 1) {
                if (n < a.N)
#pragma unroll
                    for (int j = 0; j < NCOL; ++j)
                        if (m0 + j < a.M)
                            put_out(a, static_cast<int64_t>(m0 + j) * a.N + n, Y[j]);
                continue;
            }
            // Split tile: publish this CTA's partial, count the arrival; the
            // last contributor adds all partials in CTA order and clears them.
            const int64_t slab = static_cast<int64_t>(BN) * BT;
            float *part = a.partial + (static_cast<int64_t>(tile) * a.maxc * BN + R) * BT + NCOL * ch;
            {
                float4 *dst = reinterpret_cast<float4 *>(part + (blockIdx.x - c_first) * slab);
#pragma unroll
                for (int j = 0; j < NCOL / 4; ++j)
                    put_part4(a, dst + j, make_float4(Y[4 * j], Y[4 * j + 1], Y[4 * j + 2], Y[4 * j + 3]));
            }
            __threadfence();
            named_barrier_sync(1, 256);
            if (w == 0 && lane == 0)
                *bcast = count_ok(a, tile) ? atomic_add_acq_rel_gpu(&a.count[tile], 1u) : 0u;
            named_barrier_sync(1, 256);
            const unsigned int prev = *bcast;
            if (prev == static_cast<unsigned int>(nc - 1)) {
                {
                    // this CTA's own partial is in the workspace too: Y is free
                    float *v = Y;
#pragma unroll
                    for (int j = 0; j < NCOL; ++j) v[j] = 0.0f;
                    for (int cc = 0; cc < nc; ++cc) {
                        float4 *src = reinterpret_cast<float4 *>(part + cc * slab);
#pragma unroll
                        for (int j = 0; j < NCOL / 4; ++j) {
                            const float4 p = __ldcg(src + j);
                            v[4 * j] += p.x;
                            v[4 * j + 1] += p.y;
                            v[4 * j + 2] += p.z;
                            v[4 * j + 3] += p.w;
                        }
#pragma unroll
                        for (int j = 0; j < NCOL / 4; ++j) put_part4(a, src + j, make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                    if (n < a.N)
#pragma unroll
                        for (int j = 0; j < NCOL; ++j)
                            if (m0 + j < a.M)
                                put_out(a, static_cast<int64_t>(m0 + j) * a.N + n, v[j]);
                }
                if (w == 0 && lane == 0 && count_ok(a, tile)) a.count[tile] = 0u;  // ready for the next call
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ----------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

static bool make_map(CUtensorMap *map, const void *base, CUtensorMapDataType dt, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernFn = void (*)(CUtensorMap, Args);

template <bool F16, bool CMP>
static KernFn kernel_for(int bt, int *smem)
{
    switch (bt) {
    case 16: *smem = Plan<16>::SMEM_ALLOC; return k_gemm<F16, 16, CMP>;
    case 32: *smem = Plan<32>::SMEM_ALLOC; return k_gemm<F16, 32, CMP>;
    case 64: *smem = Plan<64>::SMEM_ALLOC; return k_gemm<F16, 64, CMP>;
    default: *smem = Plan<128>::SMEM_ALLOC; return k_gemm<F16, 128, CMP>;
    }
}

static int bt_index(int bt) { return bt == 16 ? 0 : bt == 32 ? 1 : bt == 64 ? 2 : 3; }

}  // namespace gm

GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count)
{
    using namespace gm;
    GemmPlan p{};
    p.bt = 16;
    while (p.bt < 128 && p.bt < M) p.bt *= 2;
    p.mt = static_cast<int>((M + p.bt - 1) / p.bt);
    p.nt = static_cast<int>((N + BN - 1) / BN);
    const int64_t T = static_cast<int64_t>(p.mt) * p.nt;
    const int64_t NG = K / G;
    // Whole tiles in turn when every CTA gets many (the last round costs at
    // most one tile in eight); otherwise equal ranges of (tile, group) items.
    p.split = T < 8LL * sm_count && NG > 1;
    if (!p.split) {
        p.grid = static_cast<int>(T < sm_count ? T : sm_count);
        p.maxc = 1;
        p.workspace = 0;
        return p;
    }
    const int64_t items = T * NG;
    p.grid = static_cast<int>(items < sm_count ? items : sm_count);
    int maxc = 1;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t c0 = ((t * NG + 1) * p.grid - 1) / items;
        const int64_t c1 = (((t + 1) * NG) * p.grid - 1) / items;
        if (c1 - c0 + 1 > maxc) maxc = static_cast<int>(c1 - c0 + 1);
    }
    p.maxc = maxc;
    if (maxc == 1) {  // no tile is shared: the ranges fall on tile boundaries
        p.workspace = 0;
        return p;
    }
    const size_t counters = ((static_cast<size_t>(T) * sizeof(unsigned int) + 255) / 256) * 256;
    p.workspace = counters + static_cast<size_t>(T) * maxc * BN * p.bt * sizeof(float);
    return p;
}

q4_status gemm_run(const GemmPlan &p, const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                   const uint8_t *qw, bool cmp, void *y, q4_dtype yt, void *workspace,
                   unsigned int *err, uint64_t wait_ns, int debug_no_copy, cudaStream_t s,
                   cudaError_t *cerr)
{
    using namespace gm;
    *cerr = cudaSuccess;
    const bool f16 = (xt == Q4_F16);
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tmx;
    if (!make_map(&tmx, x, dt, K, M, K * 2, 64, p.bt)) return Q4_ERR_UNSUPPORTED;
    Args a{};
    a.qw = qw;
    a.y = y;
    a.yt = yt;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.mt = p.mt;
    a.nt = p.nt;
    a.split = p.split ? 1 : 0;
    a.maxc = p.maxc;
    if (p.workspace > 0) {
        const int64_t T = static_cast<int64_t>(p.mt) * p.nt;
        const size_t counters = ((static_cast<size_t>(T) * sizeof(unsigned int) + 255) / 256) * 256;
        a.count = static_cast<unsigned int *>(workspace);
        a.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + counters);
        a.count_len = T;
        a.partial_len = static_cast<int64_t>((p.workspace - counters) / sizeof(float));
    }
    a.wait_ns = wait_ns;
    a.err = err;
    a.debug_no_copy = debug_no_copy;
    int smem = 0;
    const KernFn kern = f16 ? (cmp ? kernel_for<true, true>(p.bt, &smem) : kernel_for<true, false>(p.bt, &smem))
                            : (cmp ? kernel_for<false, true>(p.bt, &smem) : kernel_for<false, false>(p.bt, &smem));
    const int variant = (cmp ? 8 : 0) + (f16 ? 4 : 0) + bt_index(p.bt);
    static std::atomic<bool> configured[16][64];  // concurrent first calls may both set it
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[variant][dev].load(std::memory_order_relaxed)) {
        *cerr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (*cerr != cudaSuccess) return Q4_ERR_CUDA;
        if (dev >= 0 && dev < 64) configured[variant][dev].store(true, std::memory_order_relaxed);
    }
    kern<<<p.grid, THREADS, smem, s>>>(tmx, a);
    *cerr = cudaGetLastError();
    return *cerr == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
