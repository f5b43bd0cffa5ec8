// gemm_tc.cu -- W4A16 GEMM on the sm_103a tcgen05 tensor cores.
//
// Y[M][N] = X[M][K] * W_hat[N][K]^T with W_hat = (q - zero) * scale per group
// of 128 along K (page "Weight quantization", "How it works"), computed the
// way the prefill path of page "LLM Quantization Architecture in Depth"
// ("Kernels and memory layout") runs: the packed codes are dequantized on
// chip into 16-bit operands and fed to the tensor cores in the same pass, so
// the floating-point weights never reach HBM.
//
// Operands.  Both MMA operands are binary16, each behind an exact power of
// two:
//     w'[n][k] = RN16(scale[n][g] * 2^-e[n] * (q - zero))
//     x'[m][k] = x[m][k] * 2^-a[m]
//     Y[m][n]  = 2^(e[n] + a[m]) * sum_k w'[n][k] x'[m][k]   (f32 accumulation)
// e[n] puts 15 * (the row's largest scale) in [2^14, 2^15), a[m] the token's
// largest |x| in the same range, so both stay inside binary16's normal range.
// x' is exact (a bf16 or f16 value has at most 11 significant bits); each w'
// is within 2^-11 (relative) of s * (q - zero).  Every term of the dot is
// therefore within 2^-11 of its exact value and the error of Y is at most
// 2^-11 * sum |w_hat x| (about 0.49e-3) plus f32 accumulation, inside the
// 1e-3 * sum |w_hat x| bound at any K and any sign pattern.  RN16(s * t)
// comes from the scale split into binary16 halves, s = hi + lo, as
// fma(hi, t, lo * t) on packed pairs (t = q - zero exact in binary16).  The
// bound holds for groups within 2^20 of their row's largest scale and token
// rows whose |x| spans less than about 2^31; beyond that binary16's
// subnormal range takes the excess precision.
//
// Passes of one call (one stream, in order):
//   1. k_prep: per weight row 2^-e[n] from its scales; per token row 2^a[m]
//      and, for bf16 activations, the binary16 copy x' in the workspace (f16
//      activations are used as they are, a[m] = 0);
//   2. k_gemm (below);
//   3. the scratch part of the workspace set back to zero.
//
// k_gemm: one persistent CTA per SM, 24 warps with fixed roles (a warp
// reaches the tensor-memory lanes of quadrant warp % 4 only and runs on SM
// partition warp % 4):
//   warp 0      activation producer: x' tiles by 2-D tensor TMA (128-byte
//               swizzle, K-major), one stage per group;
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma;
//   warp 3      weight producer: one 1-D bulk copy per step of the weight
//               layout (the tile's 8 row tiles x 4 groups, one contiguous
//               run of packed tiles) into a ring of code stages -- one copy
//               per group was measured to leave this thread, issuing eight,
//               the slowest link of the pipeline;
//   warps 4-19  operand builders in teams that take groups in turn: two
//               teams of 8 warps with 128- and 256-token tiles (a warp = one
//               k half of one lane quadrant), four teams of 4 with fewer
//               tokens (a warp = one quadrant's whole group).  Each thread owns one weight
//               row and turns its codes into packed w' pairs (shift, LOP3, one
//               packed subtraction for q - zero, one packed multiply and one
//               packed FMA per pair), stored with tcgen05.st as the MMA's A
//               operand in tensor memory.  One team alone could not keep up:
//               a group's build is a chain of waits, loads, unpacking and a
//               tensor-memory store;
//   warps 20-23 epilogue, one per quadrant: at the end of a tile each thread
//               loads its row's accumulator (tcgen05.ld), scales it by
//               2^(e[n] + a[m]) and stores it (or a partial sum, below);
//   warp 2      idle.
// Tensor memory (512 columns): the tile accumulator double-buffered in
// columns [0, 256) (one tile accumulates while the epilogue drains the
// other; a 256-token tile's single accumulator fills them, and the epilogue
// drains it before the next tile starts), four A stages of one group each at
// 256 + 64 s.  With at most 64 tokens the MMAs of each group alternate
// between two accumulators (its two k halves, summed by the epilogue): an MMA
// of fewer than 128 columns takes about 51 cycles however small, so a single
// dependent chain would leave the tensor core idle.
// A CTA tile is 128 weight rows x BT tokens, BT the smallest of 16, 32, 64,
// 128 that covers M (128 beyond; 256 when 256-token tiles alone give every
// CTA many whole tiles): 128 x BT x 16 MMAs, A from tensor memory,
// B = the activation rows from shared memory.  Per group the MMA thread waits
// for "A built and activations landed" (one builder of the team waits for the
// latter before it arrives), issues the group's 8 MMAs in one block and
// commits once, which frees the group's activation and A stage; at the end of
// a tile it commits the accumulator to the epilogue.
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
// A code stage holds one step of the weight layout: the tile's 8 row tiles x
// up to 4 groups, one contiguous run of packed tiles (row tile r, group j at
// tile r * ns + j, ns = the step's groups), fetched with one bulk copy.
constexpr int C_STAGE = RT * LB_GROUPS * TILE_BYTES;  // 35328 bytes (compact: 34304 used)
constexpr int THREADS = 24 * 32;
constexpr int W_X = 0, W_MMA = 1, W_W = 3;  // producers and the MMA thread
constexpr int W_B0 = 4, NBLD = 16;          // builders: warps 4..19
constexpr int W_E0 = 20, NEPI = 4;          // epilogue: warps 20..23
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL = 256;            // first tensor-memory column of the A stages
constexpr int NS = 4;                      // A stages (tensor memory)
constexpr int BAND = 8;                    // token tiles per raster band
// Normalizing exponents are kept in [-EMAX, EMAX]: 2^-e and 2^e stay normal
// f32 numbers.
constexpr int EMAX = 110;

template <int BT>
struct Plan {
    static constexpr int NC = BT >= 128 ? 2 : 4;  // code stages (steps of 4 groups)
    // Builder teams take groups in turn: two teams of 8 warps (one k half of
    // one lane quadrant each) with 128- and 256-token tiles, four teams of 4
    // warps (a whole group of one quadrant each) with fewer tokens.
    static constexpr int TEAMS = BT >= 128 ? 2 : 4;
    static constexpr int TEAM = NBLD / TEAMS;
    static constexpr int X_HALF = BT * 64 * 2;    // one 64-k half of a group's activations
    static constexpr int X_ST = 2 * X_HALF;
    // 256-token tiles: two activation stages (64 KB each) and one tile
    // accumulator (256 columns; the A stages take the rest of tensor
    // memory), so the epilogue drains it before the next tile starts
    static constexpr int NSX = BT >= 256 ? 2 : NS;  // activation stages
    static constexpr int NDB = BT >= 256 ? 1 : 2;   // tile accumulators
    static constexpr int OFF_X = 0;
    static constexpr int OFF_C = NSX * X_ST;
    static constexpr int OFF_BAR = ((OFF_C + NC * C_STAGE + 15) / 16) * 16;
    static constexpr int NBAR = NSX + 2 * NS + 2 * NC + 5;
    static constexpr int SMEM_USED = OFF_BAR + NBAR * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
    static_assert(X_HALF % 1024 == 0, "swizzled halves start on 1024-byte boundaries");
    static_assert(NS % TEAMS == 0, "each builder team keeps its own A stages");
    static_assert(NSX % TEAMS == 0 && NSX <= NS, "activation stages follow the A stages");
    static_assert(A_COL >= static_cast<uint32_t>(NDB * (BT > 128 ? BT : 128)), "accumulators fit below the A stages");
    static_assert(TEAM % 4 == 0, "a team covers the four lane quadrants");
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

// The 8 MMAs of one group in one block, back to back: MMA j into
// accumulator dd[j] from A columns aa[j] and B descriptor bb[j].  MMA 0 (and
// MMA 1 when TWO, the first of the second accumulator) starts a new sum
// when acc == 0; every other MMA adds.
template <bool TWO>
__device__ __forceinline__ void mma_group(const uint32_t (&dd)[8], const uint32_t (&aa)[8],
                                          const uint64_t (&bb)[8], uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p, q, t;\n\tsetp.ne.b32 p, %25, 0;\n\tsetp.ne.b32 q, %26, 0;\n\t"
        "setp.eq.b32 t, %25, %25;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %24, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [%9], %17, %24, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%2], [%10], %18, %24, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%3], [%11], %19, %24, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%4], [%12], %20, %24, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%5], [%13], %21, %24, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%6], [%14], %22, %24, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%7], [%15], %23, %24, t;\n\t"
        "}" ::"r"(dd[0]), "r"(dd[1]), "r"(dd[2]), "r"(dd[3]), "r"(dd[4]), "r"(dd[5]), "r"(dd[6]),
        "r"(dd[7]), "r"(aa[0]), "r"(aa[1]), "r"(aa[2]), "r"(aa[3]), "r"(aa[4]), "r"(aa[5]), "r"(aa[6]),
        "r"(aa[7]), "l"(bb[0]), "l"(bb[1]), "l"(bb[2]), "l"(bb[3]), "l"(bb[4]), "l"(bb[5]), "l"(bb[6]),
        "l"(bb[7]), "r"(idesc), "r"(acc), "r"(TWO ? acc : 1u)
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
__device__ __forceinline__ void tmem_ld16x(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15}, [%16];"
        : Q4_W8(v, 0), Q4_W8(v, 8)
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32x(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : Q4_W8(v, 0), Q4_W8(v, 8), Q4_W8(v, 16), Q4_W8(v, 24)
        : "r"(taddr)
        : "memory");
}
#undef Q4_R8
#undef Q4_W8

// C consecutive 32-bit columns (C = 16 or 32) of this warp's lanes.
template <int C>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[C])
{
    if constexpr (C == 16)
        tmem_ld16x(taddr, v);
    else
        tmem_ld32x(taddr, v);
}

// w' = RN16(hi * t + RN16(lo * t)) on a pair: the packed binary16 product of
// t = q - zero (exact) and the scale s = hi + lo, within 2^-11 of s * t.
__device__ __forceinline__ uint32_t scale_pair(uint32_t hi2, uint32_t lo2, uint32_t t)
{
    uint32_t p, d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(lo2), "r"(t));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(hi2), "r"(t), "r"(p));
    return d;
}

struct Args {
    const uint8_t *qw;
    void *y;
    q4_dtype yt;
    int M, N, K;
    int mt, nt;            // tiles along M (bt tokens) and N (128 rows)
    int split;             // 1: contiguous item ranges, partial sums through the workspace
    int maxc;              // most CTAs sharing one tile
    const float *rowinv;   // [N] 2^-e[n] (weight row normalization)
    const float *tokf;     // [M] 2^a[m] (token normalization), or null: 1
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

// ----------------------------------------------------------------- pass 1
// Power of two 2^p with p = (binary exponent of v) - 14, clamped to
// [-EMAX, EMAX], so that v * 2^-p lies in [2^14, 2^15); 0 when v is 0.
// `ebits` is v's biased exponent (its f32 or bf16 exponent field).
__device__ __forceinline__ int norm_exp(uint32_t ebits, bool zero)
{
    if (zero) return 0;
    const int p = static_cast<int>(ebits) - 127 - 14;  // subnormal v: clamped below
    return max(-EMAX, min(EMAX, p));
}
__device__ __forceinline__ float pow2f(int p) { return __uint_as_float(static_cast<uint32_t>(127 + p) << 23); }

// Blocks [0, row_blocks) take one 16-row weight tile per warp: the largest
// scale of each row over all its groups gives rowinv[n] = 2^-e[n], e[n] from
// 15 * max scale (the largest |q - zero| is 15).  Each later block takes one
// token row: 2^a[m] from the row's largest |x| goes to tokf[m] and, for bf16
// activations (xp not null), x * 2^-a[m] to xp as binary16 (exact: a bf16
// value keeps its 8 significant bits).  f16 activations get a[m] = 0 and are
// not copied.  A whole block per token row keeps many loads in flight when
// there are few tokens.
constexpr int PREP_THREADS = 256;
template <bool CMP>
__global__ void __launch_bounds__(PREP_THREADS) k_prep(const uint8_t *qw, int N, int K, float *rowinv,
                                                       int row_blocks, const __nv_bfloat16 *x, int M,
                                                       __half *xp, float *tokf, unsigned int *err)
{
    constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    const int lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) < row_blocks) {
        const int wid = static_cast<int>(blockIdx.x) * (PREP_THREADS / 32) + (threadIdx.x >> 5);
        const int NG = K / G;
        const int64_t ntiles = (N + TILE_ROWS - 1) / TILE_ROWS;
        if (wid >= ntiles) return;
        // scale j of a tile belongs to row (j >> 1) + 8 (j & 1)
        uint32_t mx[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) mx[j] = 0u;
#pragma unroll 2
        for (int g = lane; g < NG; g += 32) {
            const uint8_t *t = qw + tile_index(wid, g, ntiles, NG) * TBY + SCALE_OFF;
            if (CMP) {
                const uint4 h0 = *reinterpret_cast<const uint4 *>(t);
                const uint4 h1 = *reinterpret_cast<const uint4 *>(t + 16);
                const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
                    mx[2 * j] = max(mx[2 * j], __float_as_uint(fabsf(__low2float(h))));
                    mx[2 * j + 1] = max(mx[2 * j + 1], __float_as_uint(fabsf(__high2float(h))));
                }
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 f = *reinterpret_cast<const float4 *>(t + 16 * v);
                    mx[4 * v] = max(mx[4 * v], __float_as_uint(fabsf(f.x)));
                    mx[4 * v + 1] = max(mx[4 * v + 1], __float_as_uint(fabsf(f.y)));
                    mx[4 * v + 2] = max(mx[4 * v + 2], __float_as_uint(fabsf(f.z)));
                    mx[4 * v + 3] = max(mx[4 * v + 3], __float_as_uint(fabsf(f.w)));
                }
            }
        }
        uint32_t mine = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t r = __reduce_max_sync(0xffffffffu, mx[j]);
            if (lane == (j >> 1) + 8 * (j & 1)) mine = r;
        }
        const int64_t n = static_cast<int64_t>(wid) * TILE_ROWS + lane;
        if (lane < TILE_ROWS && n < N) {
            const float b = 15.0f * __uint_as_float(mine);  // largest |w_hat| of the row, bounded
            const uint32_t bits = __float_as_uint(b);
            const int e = norm_exp(min((bits >> 23) & 0xFFu, 254u), b == 0.0f);
            if (store_ok(n, N, err)) rowinv[n] = pow2f(-e);
        }
        return;
    }
    const int m = static_cast<int>(blockIdx.x) - row_blocks;
    if (m >= M) return;
    if (!xp) {  // f16 activations: used as they are
        if (threadIdx.x == 0 && store_ok(m, M, err)) tokf[m] = 1.0f;
        return;
    }
    const uint4 *row = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(m) * K);
    uint4 *out = reinterpret_cast<uint4 *>(xp + static_cast<int64_t>(m) * K);
    const int nv = K / 8;
    uint32_t amax = 0u;  // bf16 magnitude bits; their order is the order of |x|
#pragma unroll 4
    for (int v = threadIdx.x; v < nv; v += PREP_THREADS) {
        const uint4 w = row[v];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = max(amax, max(ws[j] & 0x7FFFu, (ws[j] >> 16) & 0x7FFFu));
    }
    __shared__ uint32_t red[PREP_THREADS / 32];
    amax = __reduce_max_sync(0xffffffffu, amax);
    if (lane == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < PREP_THREADS / 32; ++w) amax = max(amax, red[w]);
    const int am = norm_exp(min((amax >> 7) & 0xFFu, 254u), amax == 0u);
    const float inv = pow2f(-am);
    if (threadIdx.x == 0 && store_ok(m, M, err)) tokf[m] = pow2f(am);
#pragma unroll 4
    for (int v = threadIdx.x; v < nv; v += PREP_THREADS) {
        const uint4 w = row[v];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(ws[j] << 16) * inv;
            const float hi = __uint_as_float(ws[j] & 0xFFFF0000u) * inv;
            const __half2 h = __floats2half2_rn(lo, hi);
            o[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        if (store_ok(static_cast<int64_t>(m) * nv + v, static_cast<int64_t>(M) * nv, err))
            out[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ----------------------------------------------------------------- pass 2
// BT: tokens per tile.  CMP: compact tiles (binary16 scale pairs, zero
// nibbles, 1072 bytes).
template <int BT, bool CMP>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmx, const Args a)
{
    using P = Plan<BT>;
    constexpr int NC = P::NC, X_HALF = P::X_HALF, X_ST = P::X_ST, NSX = P::NSX, NDB = P::NDB;
    constexpr int TEAMS = P::TEAMS, TEAM = P::TEAM;
    constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    constexpr bool TWO = BT <= 64;               // two accumulators (a group's k halves)
    constexpr int CH = 16;                       // accumulator columns per tensor-memory load
    constexpr int NCH = BT / CH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sX = smem + P::OFF_X;
    uint8_t *sC = smem + P::OFF_C;
    // xfull: activations landed; afull: A built (one builder team); mdone:
    // the group's MMAs completed (frees its stages); cfull/cempty: code
    // stages (a step of up to 4 groups; every builder warp releases each);
    // dfull: a tile's accumulator complete; dempty: read by the epilogue.
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + P::OFF_BAR);
    uint64_t *xfull = bar, *afull = xfull + NSX, *mdone = afull + NS;
    uint64_t *cfull = mdone + NS, *cempty = cfull + NC;
    uint64_t *dfull = cempty + NC, *dempty = dfull + 2, *drain = dempty + 2;
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
        for (int i = 0; i < NSX; ++i) mbar_init(&xfull[i], 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(&afull[i], TEAM);
            mbar_init(&mdone[i], 1);
        }
        for (int i = 0; i < NC; ++i) {
            mbar_init(&cfull[i], 1);
            mbar_init(&cempty[i], NBLD);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], NEPI);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == W_MMA) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == W_X) {
        // ------------------------------------------------- activation producer
        if (lane == 0) {
            Cursor cur = cur0;
            int tile, g0, g1, i = 0;
            bool ok = true;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                int mb, nb;
                tile_coords(tile, a.mt, a.nt, mb, nb);
                for (int g = g0; g < g1; ++g) {
                    // stage x is free once the MMAs of group i - NSX completed
                    const int x = i % NSX, r = i - NSX;
                    if (r >= 0 && !mbar_wait_bounded(&mdone[r % NS], (r / NS) & 1, abort_flag,
                                                     a.wait_ns, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&xfull[x], static_cast<uint32_t>(X_ST));
                    uint8_t *dst = sX + x * X_ST;
                    tma_load_2d(dst, &tmx, g * G, mb * BT, &xfull[x]);
                    tma_load_2d(dst + X_HALF, &tmx, g * G + 64, mb * BT, &xfull[x]);
                    ++i;
                }
            }
            // every issued copy lands before the CTA may exit
            for (int j = max(0, i - NSX); j < i; ++j)
                mbar_wait_bounded(&xfull[j % NSX], (j / NSX) & 1, abort_flag, a.wait_ns, a.err, false);
        }
    } else if (warp == W_W) {
        // ----------------------------------------------------- weight producer
        // one bulk copy per step of the unit: the tile's row tiles x the
        // step's groups are one contiguous run of the weight layout
        if (lane == 0 && !a.debug_no_copy) {
            Cursor cur = cur0;
            int tile, g0, g1, j = 0;
            bool ok = true;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                int mb, nb;
                tile_coords(tile, a.mt, a.nt, mb, nb);
                const int rt0 = nb * RT, nrt = min(RT, ntiles_rows - rt0);
                for (int st = g0 / LB_GROUPS; st <= (g1 - 1) / LB_GROUPS; ++st, ++j) {
                    const int c = j % NC;
                    if (j >= NC && !mbar_wait_bounded(&cempty[c], ((j / NC) - 1) & 1, abort_flag,
                                                      a.wait_ns, a.err)) {
                        ok = false;
                        break;
                    }
                    const int ns = min(LB_GROUPS, NG - st * LB_GROUPS);
                    const uint32_t bytes = static_cast<uint32_t>(nrt * ns * TBY);
                    mbar_arrive_expect_tx(&cfull[c], bytes);
                    bulk_g2s(sC + c * C_STAGE,
                             a.qw + tile_index(rt0, st * LB_GROUPS, ntiles_rows, NG) * TBY, bytes,
                             &cfull[c]);
                }
            }
            for (int k = max(0, j - NC); k < j; ++k)
                mbar_wait_bounded(&cfull[k % NC], (k / NC) & 1, abort_flag, a.wait_ns, a.err, false);
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(0u, static_cast<uint32_t>(BT));
            Cursor cur = cur0;
            int tile, g0, g1, i = 0, u = 0;
            bool ok = true, issued = false;
            while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
                const int b = u % NDB;
                // the epilogue has read this accumulator's previous tile
                if (u >= NDB && !mbar_wait_bounded(&dempty[b], ((u / NDB) - 1) & 1, abort_flag,
                                                   a.wait_ns, a.err, true, true)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem + static_cast<uint32_t>(b) * 128u;
                for (int g = g0; g < g1; ++g, ++i) {
                    const int s = i % NS;
                    // A built and activations landed
                    if (!mbar_wait_bounded(&afull[s], (i / NS) & 1, abort_flag, a.wait_ns, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // one descriptor per stage; a k step's operand lies a
                    // constant number of 16-byte units further on
                    const uint64_t xd = sw128_desc(smem_u32(sX + (i % NSX) * X_ST));
                    const uint32_t at = tmem + A_COL + static_cast<uint32_t>(s) * 64u;
                    const uint32_t acc = g > g0 ? 1u : 0u;  // the tile's first k step starts the sum
                    uint32_t dd[8], aa[8];
                    uint64_t bb[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // TWO: k step k of half h is MMA 2k + h into accumulator h
                        const int k16 = TWO ? 4 * (j & 1) + (j >> 1) : j;
                        dd[j] = TWO ? d + 64u * (j & 1) : d;
                        aa[j] = at + 8u * k16;
                        bb[j] = xd + ((k16 >> 2) * X_HALF + 32 * (k16 & 3)) / 16;
                    }
                    mma_group<TWO>(dd, aa, bb, idesc, acc);
                    issued = true;
                    mma_commit(&mdone[s]);
                }
                if (!ok) break;
                mma_commit(&dfull[b]);
                ++u;
            }
            if (issued) {
                // all issued MMAs complete before tensor memory is freed
                mma_commit(drain);
                mbar_wait_bounded(drain, 0, abort_flag, a.wait_ns, a.err, false);
            }
        }
    } else if (warp >= W_B0 && warp < W_B0 + NBLD) {
        // ------------------------------------------------ A operand builders
        // The teams build groups in turn (team = group index % TEAMS), so
        // that TEAMS groups are in the making at once: one group's build is
        // a chain of waits, shared-memory loads, unpacking and a
        // tensor-memory store that one team cannot shorten.  Each team uses
        // its own A stages (NS % TEAMS == 0).
        // Thread = weight row R of the tile (tensor-memory lane R); warp w of
        // a team (w % 4 = q) builds lane quadrant q, k half kh (two teams) or
        // both halves (four teams): the k steps 4 kh .. 4 kh + 3 of the
        // group, tensor-memory columns 32 kh .. 32 kh + 31 of the A stage.
        // The row's codes sit in lanes 4 (R % 8) + t of its packed tile
        // (t = 0..3), in the nibble fields of row R % 16 (tiled layout,
        // include/q4.h): word i of chunk h of lane 4 (R % 8) + t holds
        // k = 16 (4h + i) + 2t + {0, 1} and + {8, 9}, i.e. A columns
        // 8 (4h + i) + t and 8 (4h + i) + t + 4.
        const int team = (warp - W_B0) / TEAM, wt = (warp - W_B0) % TEAM;
        const int q = warp & 3;
        const int kh0 = TEAMS == 2 ? wt >> 2 : 0, kh1 = TEAMS == 2 ? kh0 + 1 : 2;
        const int R = 32 * q + lane, d = R >> 4, rr = R & 15;
        const int lg = 4 * (rr & 7);
        const uint32_t sA = (rr & 8) ? 4u : 0u, sB = (rr & 8) ? 8u : 12u;
        const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q) << 16) + A_COL;
        Cursor cur = cur0;
        int tile, g0, g1, i = 0, j = 0;
        bool ok = true;
        while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
            int mb, nb;
            tile_coords(tile, a.mt, a.nt, mb, nb);
            const int nrt = min(RT, ntiles_rows - nb * RT);
            const int n = nb * BN + R;
            const bool live = d < nrt;
            // rows past the matrix inside the last tile carry zero codes and scales
            const float rinv = (live && n < a.N) ? a.rowinv[n] : 0.0f;
            for (int g = g0; ok && g < g1; ++j) {
                // step st of the unit: code stage c; every builder warp waits
                // for it and releases it, whether or not its team builds one
                // of the step's groups
                const int st = g / LB_GROUPS, c = j % NC;
                const int ns = min(LB_GROUPS, NG - st * LB_GROUPS), gend = min(g1, st * LB_GROUPS + ns);
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&cfull[c], (j / NC) & 1, abort_flag,
                                                               a.wait_ns, a.err));
                for (; ok && g < gend; ++g, ++i) {
                if ((i & (TEAMS - 1)) != team) continue;
                const int s = i % NS;
                // A stage s is free once the MMAs of group i - NS completed
                if (i >= NS)
                    ok = mbar_wait_bounded(&mdone[s], ((i / NS) - 1) & 1, abort_flag, a.wait_ns,
                                           a.err);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const uint8_t *ct = sC + c * C_STAGE + (d * ns + (g - st * LB_GROUPS)) * TBY;
                uint32_t hi2 = 0u, lo2 = 0u, mz = 0u;
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
                    // s' = s * 2^-e[n] (exact), split into binary16 hi + lo
                    const float sp = sc * rinv;
                    const __half hi = __float2half_rn(sp);
                    const __half lo = __float2half_rn(sp - __half2float(hi));
                    const __half2 hi2h = __halves2half2(hi, hi), lo2h = __halves2half2(lo, lo);
                    hi2 = *reinterpret_cast<const uint32_t *>(&hi2h);
                    lo2 = *reinterpret_cast<const uint32_t *>(&lo2h);
                    const __half2 mzh = __floats2half2_rn(-(1024.0f + z), -(1024.0f + z));
                    mz = *reinterpret_cast<const uint32_t *>(&mzh);  // exact
                }
#pragma unroll 1
                for (int kh = kh0; kh < kh1; ++kh) {
                    uint32_t v[32];
                    if (live) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const uint4 w4 = *reinterpret_cast<const uint4 *>(ct + kh * 512 + 16 * (lg + t));
                            const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                const uint32_t ta = sub_pair<true>(lop3_and_or(ws[jj] >> sA, 0x000F000Fu, 0x64006400u), mz);
                                const uint32_t tb = sub_pair<true>(lop3_and_or(ws[jj] >> sB, 0x000F000Fu, 0x64006400u), mz);
                                v[8 * jj + t] = scale_pair(hi2, lo2, ta);
                                v[8 * jj + t + 4] = scale_pair(hi2, lo2, tb);
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;  // row tiles past the matrix
                    }
                    tmem_st32(tlane + static_cast<uint32_t>(s) * 64u + 32u * kh, v);
                }
                tmem_wait_st();
                tc_fence_before();
                // one builder of the team also waits for the stage's
                // activations, so that A built = everything the MMAs of
                // group i read is in place
                bool landed = true;
                if (wt == 0)
                    landed = mbar_wait_bounded(&xfull[i % NSX], (i / NSX) & 1, abort_flag, a.wait_ns,
                                               a.err);
                __syncwarp();
                if (!__all_sync(0xffffffffu, landed)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive(&afull[s]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&cempty[c]);
            }
        }
    } else if (warp >= W_E0) {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3, R = 32 * q + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        Cursor cur = cur0;
        int tile, g0, g1, u = 0;
        bool ok = true;
        while (ok && next_unit(a, NG, cur, tile, g0, g1)) {
            const int b = u % NDB;
            int mb, nb;
            tile_coords(tile, a.mt, a.nt, mb, nb);
            const int n = nb * BN + R;
            const float fn = n < a.N ? __frcp_rn(a.rowinv[n]) : 0.0f;  // 2^e[n], exact
            ok = mbar_wait_bounded(&dfull[b], (u / NDB) & 1, abort_flag, a.wait_ns, a.err);
            ok = __all_sync(0xffffffffu, ok);
            const int64_t first = static_cast<int64_t>(tile) * NG;
            int c_first = blockIdx.x, nc = 1;
            if (a.split) {
                c_first = static_cast<int>(owner_of(first, items, gridDim.x));
                nc = static_cast<int>(owner_of(first + NG - 1, items, gridDim.x)) - c_first + 1;
                // every epilogue warp decides together whether to go on
                if (named_barrier_or(1, 32 * NEPI, !ok)) {
                    ok = false;
                    break;
                }
            } else if (!ok) {
                break;
            }
            tc_fence_after();
            const uint32_t db = tl + static_cast<uint32_t>(b) * 128u;
            const int m0 = mb * BT;
            const int64_t slab = static_cast<int64_t>(BN) * BT;
            float *part = a.partial + (static_cast<int64_t>(tile) * a.maxc * BN + R) * BT;
#pragma unroll 1
            for (int cc = 0; cc < NCH; ++cc) {
                uint32_t v[CH];
                tmem_ld<CH>(db + cc * CH, v);
                if constexpr (TWO) {
                    uint32_t w[CH];
                    tmem_ld<CH>(db + 64u + cc * CH, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(w[j]));
                } else {
                    tmem_wait_ld();
                }
                if (cc == NCH - 1) {  // the accumulator is read: the next tile may use it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dempty[b]);
                }
                if (nc == 1) {
                    if (n < a.N)
#pragma unroll
                        for (int j = 0; j < CH; ++j) {
                            const int m = m0 + cc * CH + j;
                            if (m < a.M) {
                                const float tf = a.tokf ? __ldg(a.tokf + m) : 1.0f;
                                put_out(a, static_cast<int64_t>(m) * a.N + n,
                                        __uint_as_float(v[j]) * fn * tf);
                            }
                        }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(part + (blockIdx.x - c_first) * slab + cc * CH);
#pragma unroll
                    for (int j = 0; j < CH / 4; ++j)
                        put_part4(a, dst + j,
                                  make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                              __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
                }
            }
            ++u;
            if (nc == 1) continue;
            // Split tile: count this CTA's arrival; the last contributor adds
            // all partials in CTA order, clears them and stores the tile.
            __threadfence();
            named_barrier_sync(1, 32 * NEPI);
            if (warp == W_E0 && lane == 0)
                *bcast = count_ok(a, tile) ? atomic_add_acq_rel_gpu(&a.count[tile], 1u) : 0u;
            named_barrier_sync(1, 32 * NEPI);
            const unsigned int prev = *bcast;
            if (prev != static_cast<unsigned int>(nc - 1)) continue;
#pragma unroll 1
            for (int cc = 0; cc < NCH; ++cc) {
                float sum[CH];
#pragma unroll
                for (int j = 0; j < CH; ++j) sum[j] = 0.0f;
                for (int k = 0; k < nc; ++k) {
                    float4 *src = reinterpret_cast<float4 *>(part + k * slab + cc * CH);
#pragma unroll
                    for (int j = 0; j < CH / 4; ++j) {
                        const float4 p = __ldcg(src + j);
                        sum[4 * j] += p.x;
                        sum[4 * j + 1] += p.y;
                        sum[4 * j + 2] += p.z;
                        sum[4 * j + 3] += p.w;
                    }
#pragma unroll
                    for (int j = 0; j < CH / 4; ++j) put_part4(a, src + j, make_float4(0.f, 0.f, 0.f, 0.f));
                }
                if (n < a.N)
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int m = m0 + cc * CH + j;
                        if (m < a.M) {
                            const float tf = a.tokf ? __ldg(a.tokf + m) : 1.0f;
                            put_out(a, static_cast<int64_t>(m) * a.N + n, sum[j] * fn * tf);
                        }
                    }
            }
            if (warp == W_E0 && lane == 0 && count_ok(a, tile)) a.count[tile] = 0u;  // ready for the next call
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) tmem_dealloc(tmem, TMEM_COLS);
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

template <bool CMP>
static KernFn kernel_for(int bt, int *smem)
{
    switch (bt) {
    case 16: *smem = Plan<16>::SMEM_ALLOC; return k_gemm<16, CMP>;
    case 32: *smem = Plan<32>::SMEM_ALLOC; return k_gemm<32, CMP>;
    case 64: *smem = Plan<64>::SMEM_ALLOC; return k_gemm<64, CMP>;
    case 128: *smem = Plan<128>::SMEM_ALLOC; return k_gemm<128, CMP>;
    default: *smem = Plan<256>::SMEM_ALLOC; return k_gemm<256, CMP>;
    }
}

static int bt_index(int bt) { return bt == 16 ? 0 : bt == 32 ? 1 : bt == 64 ? 2 : bt == 128 ? 3 : 4; }

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: [0, zero) split-K counters and partial sums (left zero by every
// completed call), then the scratch of pass 1 (also set back to zero):
// rowinv [N] f32, tokf [M] f32, x' [M][K] binary16.
struct Scratch {
    size_t zero, rows, tok, xp, end;
};
static Scratch scratch_layout(const GemmPlan &p, int64_t M, int64_t N, int64_t K, size_t zero)
{
    Scratch s;
    s.zero = zero;
    s.rows = align_up(zero, 1024);
    s.tok = s.rows + align_up(static_cast<size_t>(N) * 4, 1024);
    s.xp = s.tok + align_up(static_cast<size_t>(M) * 4, 1024);
    s.end = s.xp + static_cast<size_t>(M) * K * 2;
    (void)p;
    return s;
}

static size_t zero_bytes(const GemmPlan &p)
{
    if (!p.split || p.maxc == 1) return 0;
    const int64_t T = static_cast<int64_t>(p.mt) * p.nt;
    const size_t counters = align_up(static_cast<size_t>(T) * sizeof(unsigned int), 256);
    return counters + static_cast<size_t>(T) * p.maxc * BN * p.bt * sizeof(float);
}

}  // namespace gm

GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count)
{
    using namespace gm;
    GemmPlan p{};
    p.bt = 16;
    while (p.bt < 128 && p.bt < M) p.bt *= 2;
    p.nt = static_cast<int>((N + BN - 1) / BN);
    // 256-token tiles (twice the MMA work per group built) only when they
    // alone give every CTA many whole tiles: split over CTAs, their single
    // accumulator stalls at every short unit (measured 35% slower there)
    if (M > 128 && ((M + 255) / 256) * p.nt >= 8LL * sm_count) p.bt = 256;
    p.mt = static_cast<int>((M + p.bt - 1) / p.bt);
    const int64_t T = static_cast<int64_t>(p.mt) * p.nt;
    const int64_t NG = K / G;
    // Whole tiles in turn when every CTA gets many (the last round costs at
    // most one tile in eight); otherwise equal ranges of (tile, group) items.
    p.split = T < 8LL * sm_count && NG > 1;
    p.maxc = 1;
    if (!p.split) {
        p.grid = static_cast<int>(T < sm_count ? T : sm_count);
    } else {
        const int64_t items = T * NG;
        p.grid = static_cast<int>(items < sm_count ? items : sm_count);
        int maxc = 1;
        for (int64_t t = 0; t < T; ++t) {
            const int64_t c0 = ((t * NG + 1) * p.grid - 1) / items;
            const int64_t c1 = (((t + 1) * NG) * p.grid - 1) / items;
            if (c1 - c0 + 1 > maxc) maxc = static_cast<int>(c1 - c0 + 1);
        }
        p.maxc = maxc;  // 1: the ranges fall on tile boundaries, no tile is shared
    }
    p.workspace = scratch_layout(p, M, N, K, zero_bytes(p)).end;
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
    const Scratch sl = scratch_layout(p, M, N, K, zero_bytes(p));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *rowinv = reinterpret_cast<float *>(ws + sl.rows);
    float *tokf = reinterpret_cast<float *>(ws + sl.tok);
    __half *xp = reinterpret_cast<__half *>(ws + sl.xp);

    // pass 1: row and token normalizations, the binary16 copy of bf16 activations
    const int64_t row_tiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int row_blocks = static_cast<int>((row_tiles + PREP_THREADS / 32 - 1) / (PREP_THREADS / 32));
    const int prep_blocks = static_cast<int>(row_blocks + M);
    const auto *xb = static_cast<const __nv_bfloat16 *>(f16 ? nullptr : x);
    if (cmp)
        k_prep<true><<<prep_blocks, PREP_THREADS, 0, s>>>(qw, static_cast<int>(N), static_cast<int>(K),
                                                          rowinv, row_blocks, xb, static_cast<int>(M),
                                                          f16 ? nullptr : xp, tokf, err);
    else
        k_prep<false><<<prep_blocks, PREP_THREADS, 0, s>>>(qw, static_cast<int>(N), static_cast<int>(K),
                                                           rowinv, row_blocks, xb, static_cast<int>(M),
                                                           f16 ? nullptr : xp, tokf, err);
    *cerr = cudaGetLastError();
    if (*cerr != cudaSuccess) return Q4_ERR_CUDA;

    // pass 2
    CUtensorMap tmx;
    if (!make_map(&tmx, f16 ? x : static_cast<const void *>(xp), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, K,
                  M, K * 2, 64, p.bt))
        return Q4_ERR_UNSUPPORTED;
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
    a.rowinv = rowinv;
    a.tokf = f16 ? nullptr : tokf;
    if (sl.zero > 0) {
        const int64_t T = static_cast<int64_t>(p.mt) * p.nt;
        const size_t counters = align_up(static_cast<size_t>(T) * sizeof(unsigned int), 256);
        a.count = reinterpret_cast<unsigned int *>(ws);
        a.partial = reinterpret_cast<float *>(ws + counters);
        a.count_len = T;
        a.partial_len = static_cast<int64_t>((sl.zero - counters) / sizeof(float));
    }
    a.wait_ns = wait_ns;
    a.err = err;
    a.debug_no_copy = debug_no_copy;
    int smem = 0;
    const KernFn kern = cmp ? kernel_for<true>(p.bt, &smem) : kernel_for<false>(p.bt, &smem);
    const int variant = (cmp ? 5 : 0) + bt_index(p.bt);
    static std::atomic<bool> configured[10][64];  // concurrent first calls may both set it
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[variant][dev].load(std::memory_order_relaxed)) {
        *cerr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (*cerr != cudaSuccess) return Q4_ERR_CUDA;
        if (dev >= 0 && dev < 64) configured[variant][dev].store(true, std::memory_order_relaxed);
    }
    kern<<<p.grid, THREADS, smem, s>>>(tmx, a);
    *cerr = cudaGetLastError();
    if (*cerr != cudaSuccess) return Q4_ERR_CUDA;

    // pass 3: the scratch written by pass 1 back to zero
    *cerr = cudaMemsetAsync(ws + sl.rows, 0, (f16 ? sl.xp : sl.end) - sl.rows, s);
    return *cerr == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
