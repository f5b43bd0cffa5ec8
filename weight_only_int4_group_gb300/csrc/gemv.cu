// gemv.cu -- decode W4A16 GEMV for 1 <= M <= 16 on sm_103a.
//
// Computes y[m][n] = sum over groups g of
//     scale[n][g] * (sum_{k in g} q[n][k] * x[m][k] - zero[n][g] * sum_{k in g} x[m][k])
// i.e. the factored group dot of the page "Weight quantization" (tirogla.com,
// sections "How it works" and "Code", function `dot`), with the 4-bit codes
// turned into floating point in registers and never written back to memory.
//
// Work decomposition (stream-K): the output rows are cut into row blocks of
// RB = 8 tiles (128 rows; 4 tiles when 9 <= M <= 16 and 8-tile blocks would
// give each CTA fewer than 8 steps); each row block is a sequence of
// NS = ceil(NG/4) steps, a step being 4 consecutive groups along K (one
// contiguous run of the weight layout's tiles).  The nrb * NS items are
// split into `grid` contiguous, equal ranges, one per persistent CTA (two
// CTAs per SM).  A CTA accumulates the steps of a row block in registers and
// writes the row block out when it reaches its last step; a row block whose
// steps are spread over several CTAs is finished by the last of them to
// arrive, which sums the partial results in CTA order (so results do not
// depend on timing).
//
// Consecutive GEMVs on a stream overlap (programmatic dependent launch): each
// kernel lets the next launch at once, and the next one's producer requests
// its first stages of weight tiles before waiting for the previous kernel to
// complete; activations, outputs and the workspace are touched only after.
//
// CTA = 4 consumer warps + 1 producer warp + 1 epilogue warp.  The producer
// streams each step's weight tiles (RB row tiles x 4 groups) with 1-D bulk
// asynchronous copies (TMA engine) into a 2-stage shared-memory ring and runs
// ahead across row blocks, so the memory pipeline never drains.  Consumer
// warp w takes group w of every step.  When the consumers finish their share
// of a row block they sum it over the warps into a shared-memory hand-off
// buffer and go straight on to the next step; the epilogue warp writes the
// rows out (or the partial sums, then the arrival counter and, if it arrives
// last, the final sum), so global-memory round trips never stall the
// consumers.
//
// Two consumer variants:
//   FMA (M = 1): CUDA-core path.  A 4-bit code q at bit offset 16 or 12 of a
//     word becomes the f32 value 1 + q/128 or 1 + q/2048 with one LOP3
//     (mantissa bits under the exponent of 1.0); two such values are
//     multiplied into a pair of f32 accumulators by one packed FFMA2.  The
//     constant 1 is removed per group with the activation sums.  The step's
//     activations ride in the same stage; each warp turns its group's into
//     the per-lane pair order.
//   MMA (M = 1..16, bf16/f16 activations; f32 activations as bf16 hi + lo):
//     each word yields the four A-fragment registers of an m16n8k16
//     tensor-core MMA as bf16 pairs 128 + q (f16: 1024 + q) with one LOP3
//     each; the activations are the B fragment (the batch is the MMA's n
//     dimension).  For M <= 8 (bf16/f16) the producer copies the step's
//     activation rows (f32 at M = 1 for f32 activations, split into hi + lo
//     per step) into the stage next to the tiles (rows padded by 16
//     bytes so the eight batch rows fall in different banks); otherwise each
//     lane loads its B fragments from L2 one step ahead.  The group sums of the
//     activations come from one extra MMA per k-step with an all-ones A
//     operand.  Per group, y += scale * (D - (offset + zero) * sum x).
//
//   Row-split MMA (9 <= M <= 16, bf16/f16 activations): consumer warp w
//     takes row tiles w * RB/4 .. of every step, all 4 groups, so a row
//     block needs no reduction across warps and a warp keeps 4x fewer
//     accumulators; the step's activation rows (up to 16) are staged with
//     the tiles and read as B fragments with ldmatrix (rows padded by 16
//     bytes: conflict-free).  The A operand is the small integer q - zero
//     itself (offset + q from the LOP3, minus offset + zero with one packed
//     FMA, exact in bf16/f16), so no activation sums are needed: per group
//     y += scale * D, a fifth fewer MMAs than with activation sums.  For
//     2 <= M <= 8 the group-split MMA consumer above is faster (measured
//     3-11% per launch and 1-10% on the 70B decode step).
//
// Both consumers read 1104-byte tiles (f32 scales, u8 zeros); the tensor-core
// one also reads compact 1072-byte tiles (binary16 scales widened exactly,
// zero nibbles; the format the page "Weight quantization" counts as 16-bit
// scales and 4-bit zeros), selected at compile time.
#include <mutex>
#include <unordered_map>

#include "common.cuh"

namespace q4 {

constexpr int W = 4;        // consumer warps = groups per step
constexpr int RB = 8;       // row tiles per row block (RB_SMALL_ROWS for small problems)
constexpr int RB_SMALL_ROWS = 4;  // small problems, row-split consumers (one tile per warp)
constexpr int NSTAGE = 2;   // ring depth (3 for the M = 1 tensor-core kernel on long runs)
constexpr int THREADS = (W + 2) * 32;  // consumers, producer, epilogue
constexpr int CONSUMERS = W * 32;
constexpr int XSTAGE_BYTES = W * G * 4;           // FMA: the step's activations (f32 worst case)
constexpr int CTRL_BYTES = 256;                   // barriers + flags (rings up to 15 stages)
// FMA activation pairs, per warp: one record of 64 floats per lane class t,
// padded to 68 floats so the four lane classes read four different bank
// groups in one wavefront; then the four sum records.
constexpr int PAIR_STRIDE = 68;
constexpr int WARP_PAIR_FLOATS = 4 * PAIR_STRIDE + 4 * 4;
constexpr int MIN_BLOCKS = 2;  // CTAs per SM the shared memory budget is sized for

constexpr int XROW = W * G * 2 + 16;  // MMA staged activations: one padded row per batch row
// a step is one step of the weight layout's blocks, and a row block lies in
// one layout block: the tiles of an item are one contiguous run
static_assert(W == LB_GROUPS && LB_TILES % RB == 0 && LB_TILES % RB_SMALL_ROWS == 0,
              "row blocks and steps nest in the weight layout's blocks");

// xrows: batch rows staged with each step (MMA, M <= 8); 0 otherwise;
// tb: bytes per tile (TILE_BYTES, or CMP_TILE_BYTES for compact metadata)
__host__ __device__ constexpr int stage_bytes(int mode, int xrows, int rb = RB, int tb = TILE_BYTES)
{
    return mode == PATH_FMA ? rb * W * tb + XSTAGE_BYTES
                            : ((rb * W * tb + xrows * XROW + 127) / 128) * 128;
}

__host__ __device__ constexpr int smem_bytes(int mode, int xrows, int ms, int nstage = NSTAGE,
                                             int rb = RB, int tb = TILE_BYTES)
{
    return nstage * stage_bytes(mode, xrows, rb, tb) + CTRL_BYTES +
           (mode == PATH_FMA ? (W * WARP_PAIR_FLOATS + W * rb * 16) * 4 : W * rb * 16 * ms * 4) +
           rb * 16 * ms * 4;  // hand-off buffer of one row block
}


static_assert(MIN_BLOCKS * (smem_bytes(PATH_FMA, 0, 1) + 1024) <= 228 * 1024, "two FMA CTAs per SM");
static_assert(MIN_BLOCKS * (smem_bytes(PATH_MMA, 8, 8) + 1024) <= 228 * 1024, "two MMA CTAs per SM");
static_assert(MIN_BLOCKS * (smem_bytes(PATH_MMA, 0, 16) + 1024) <= 228 * 1024, "two MMA CTAs per SM");
static_assert(MIN_BLOCKS * (NSTAGE * stage_bytes(PATH_MMA, 16) + CTRL_BYTES + RB * 16 * 16 * 4 + 1024) <=
                  228 * 1024,
              "two row-split CTAs per SM at M = 16");
static_assert(MIN_BLOCKS * (smem_bytes(PATH_MMA, 1, 1, 3) + 1024) <= 228 * 1024,
              "two 3-stage M = 1 MMA CTAs per SM");

__device__ __forceinline__ void store_y(void *y, q4_dtype yt, int64_t idx, float v)
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
__device__ __forceinline__ void put_y(const GemvArgs &a, int64_t idx, float v)
{
    if (store_ok(idx, static_cast<int64_t>(a.M) * a.N, a.err)) store_y(a.y, a.yt, idx, v);
}
__device__ __forceinline__ void put_part(const GemvArgs &a, float *p, float v)
{
    if (store_ok(p - a.partial, a.partial_len, a.err)) *p = v;
}
__device__ __forceinline__ void put_part4(const GemvArgs &a, float4 *p, float4 v)
{
    if (store_ok(reinterpret_cast<float *>(p) - a.partial + 3, a.partial_len, a.err)) *p = v;
}
__device__ __forceinline__ bool count_ok(const GemvArgs &a, int rb)
{
    return store_ok(rb, a.count_len, a.err);
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

// Four 8x8 b16 matrices from shared memory; thread 8i + r gives row r of
// matrix i, and thread 4g + t receives elements (g, 2t) and (g, 2t + 1) of
// each: with the activation rows as matrix rows these are B fragments.
__device__ __forceinline__ void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                            const void *row_addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(row_addr)));
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


// One word -> the four A-fragment registers (bf16 128 + q or f16 1024 + q
// pairs: one shift and one LOP3 each) -> one m16n8k16 MMA into d.  Written as
// a single PTX block so the fragment registers are allocated in place.
template <int ABT>
__device__ __forceinline__ void mma_word(float (&d)[4], uint32_t w, uint32_t b0, uint32_t b1)
{
    if (ABT == 0)
        asm("{\n\t.reg .b32 t1, t2, t3, a0, a1, a2, a3;\n\t"
            "shr.b32 t1, %4, 4;\n\tshr.b32 t2, %4, 8;\n\tshr.b32 t3, %4, 12;\n\t"
            "lop3.b32 a0, %4, 0x000F000F, 0x43004300, 0xEA;\n\t"
            "lop3.b32 a1, t1, 0x000F000F, 0x43004300, 0xEA;\n\t"
            "lop3.b32 a3, t2, 0x000F000F, 0x43004300, 0xEA;\n\t"
            "lop3.b32 a2, t3, 0x000F000F, 0x43004300, 0xEA;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%5,%6}, {%0,%1,%2,%3};\n\t}"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(w), "r"(b0), "r"(b1));
    else
        asm("{\n\t.reg .b32 t1, t2, t3, a0, a1, a2, a3;\n\t"
            "shr.b32 t1, %4, 4;\n\tshr.b32 t2, %4, 8;\n\tshr.b32 t3, %4, 12;\n\t"
            "lop3.b32 a0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
            "lop3.b32 a1, t1, 0x000F000F, 0x64006400, 0xEA;\n\t"
            "lop3.b32 a3, t2, 0x000F000F, 0x64006400, 0xEA;\n\t"
            "lop3.b32 a2, t3, 0x000F000F, 0x64006400, 0xEA;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3}, {%5,%6}, {%0,%1,%2,%3};\n\t}"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(w), "r"(b0), "r"(b1));
}

// One word (and the next word of its 16-byte chunk, for the funnel step) ->
// four packed FFMA2 steps: code pairs from bit offsets (16, 12) of w, w >> 8,
// w << 8 and the funnel (w_next:w) >> 16, each made with two LOP3s.
__device__ __forceinline__ void fma_word(float2 &aG, float2 &aG8, uint32_t w, uint32_t wn,
                                         float2 p0, float2 p1, float2 p2, float2 p3)
{
    asm("{\n\t.reg .b32 r8, l8, fu, l, h;\n\t.reg .b64 v, x, g, g8;\n\t"
        "mov.b64 g, {%0, %1};\n\tmov.b64 g8, {%2, %3};\n\t"
        "shr.b32 r8, %4, 8;\n\tshl.b32 l8, %4, 8;\n\tshf.r.clamp.b32 fu, %4, %5, 16;\n\t"
        "lop3.b32 l, %4, 0x000F0000, 0x3F800000, 0xEA;\n\tlop3.b32 h, %4, 0x0000F000, 0x3F800000, 0xEA;\n\t"
        "mov.b64 v, {l, h};\n\tmov.b64 x, {%6, %7};\n\tfma.rn.f32x2 g, v, x, g;\n\t"
        "lop3.b32 l, r8, 0x000F0000, 0x3F800000, 0xEA;\n\tlop3.b32 h, r8, 0x0000F000, 0x3F800000, 0xEA;\n\t"
        "mov.b64 v, {l, h};\n\tmov.b64 x, {%8, %9};\n\tfma.rn.f32x2 g8, v, x, g8;\n\t"
        "lop3.b32 l, l8, 0x000F0000, 0x3F800000, 0xEA;\n\tlop3.b32 h, l8, 0x0000F000, 0x3F800000, 0xEA;\n\t"
        "mov.b64 v, {l, h};\n\tmov.b64 x, {%10, %11};\n\tfma.rn.f32x2 g8, v, x, g8;\n\t"
        "lop3.b32 l, fu, 0x000F0000, 0x3F800000, 0xEA;\n\tlop3.b32 h, fu, 0x0000F000, 0x3F800000, 0xEA;\n\t"
        "mov.b64 v, {l, h};\n\tmov.b64 x, {%12, %13};\n\tfma.rn.f32x2 g, v, x, g;\n\t"
        "mov.b64 {%0, %1}, g;\n\tmov.b64 {%2, %3}, g8;\n\t}"
        : "+f"(aG.x), "+f"(aG.y), "+f"(aG8.x), "+f"(aG8.y)
        : "r"(w), "r"(wn), "f"(p0.x), "f"(p0.y), "f"(p1.x), "f"(p1.y), "f"(p2.x), "f"(p2.y),
          "f"(p3.x), "f"(p3.y));
}

// First item of CTA c, and the CTA that owns item i, for T items over G CTAs.
__host__ __device__ __forceinline__ int64_t range_begin(int64_t c, int64_t T, int64_t G)
{
    return c * T / G;
}
__host__ __device__ __forceinline__ int64_t owner_of(int64_t i, int64_t T, int64_t G)
{
    return ((i + 1) * G - 1) / T;
}

// Scale and zero pairs (rows i and i + 8 of a tile, i = gq) of one tile:
// f32 scales and u8 zeros, or (compact) binary16 scales and one byte of two
// zero nibbles; the zeros come back as z_i | z_{i+8} << 8 either way.
template <bool CMP>
__device__ __forceinline__ void tile_meta(const uint8_t *tile, int gq, float2 &sp, uint32_t &zp)
{
    if (CMP) {
        sp = __half22float2(*reinterpret_cast<const __half2 *>(tile + SCALE_OFF + 4 * gq));
        const uint32_t b = tile[CMP_ZERO_OFF + gq];
        zp = (b & 0x0Fu) | ((b >> 4) << 8);
    } else {
        sp = *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq);
        zp = *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq);
    }
}


// Row-split consumer loop (see the file header): warp w accumulates row tiles
// TPW w .. TPW w + TPW - 1 of each row block over all W groups of a step.
template <int NT, int ABT, int NSTG, int RBT, bool CMP>
__device__ __forceinline__ void consume_rows(const GemvArgs &a, uint8_t *ring, int SB, uint64_t *full,
                                             uint64_t *empty, uint64_t *ofull, uint64_t *ofree,
                                             volatile int *abort_flag, float *out, int64_t beg,
                                             int64_t end, int NS, int ntiles, int NG)
{
    constexpr int RB = RBT, TPW = RBT / W;
    constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    constexpr int TILES_BYTES = RBT * W * TBY;
    const uint32_t MAG = ABT == 0 ? 0x43004300u : 0x64006400u;  // offset + q: 128 + q or 1024 + q
    const uint32_t NEG = ABT == 0 ? 0xC300C300u : 0xE400E400u;  // -(offset + zero), zero in the low bits
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, t = lane & 3;
    const int M = a.M;
    // ldmatrix: this lane gives row (token) lm_tok of matrix lm_mat; matrix
    // i holds k = 16 (j + i / 2) + 8 (i % 2) .. + 7 of k-step pair (j, j + 1)
    const int lm_tok = lane & 7, lm_mat = lane >> 3;
    int xoff[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int tok = min(8 * n + lm_tok, M - 1);  // rows past M: never stored
        xoff[n] = tok * XROW + (16 * (lm_mat >> 1) + 8 * (lm_mat & 1)) * 2;
    }
    float yacc[TPW][NT][4];
    int gstep = 0, nepi = 0;
    int rb = static_cast<int>(beg / NS), s = static_cast<int>(beg % NS) - 1;
    for (int64_t it = beg; it < end; ++it, ++gstep) {
        if (++s == NS) {
            s = 0;
            ++rb;
        }
        const int slot = gstep % NSTG;
        if (it == beg || s == 0) {
#pragma unroll
            for (int r = 0; r < TPW; ++r)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) yacc[r][n][e] = 0.0f;
        }
        const bool ok = mbar_wait_bounded(&full[slot], (gstep / NSTG) & 1, abort_flag, a.wait_ns, a.err);
        if (!__all_sync(0xffffffffu, ok)) return;
        const uint8_t *stage = ring + slot * SB;
        const uint8_t *xs = stage + TILES_BYTES;
        // GP groups at a time (two at once measured slower at one batch tile,
        // and two batch tiles have no registers to spare)
        constexpr int GP = 1;
#pragma unroll 1
        for (int gi0 = 0; gi0 < W; gi0 += GP) {
            if (s * W + gi0 >= NG) break;  // the last step may hold fewer groups
            // B fragments of the groups' 8 k-steps for every batch tile; a
            // group past K (odd group count) reads the stage's bytes and is
            // discarded
            uint32_t bf[GP][NT][8][2];
#pragma unroll
            for (int gp = 0; gp < GP; ++gp)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        ldmatrix_x4(bf[gp][n][2 * jj][0], bf[gp][n][2 * jj][1], bf[gp][n][2 * jj + 1][0],
                                    bf[gp][n][2 * jj + 1][1], xs + xoff[n] + (gi0 + gp) * G * 2 + jj * 64);
            // this warp's row tiles of the groups: codes, scales and the
            // packed -(offset + zero) of rows g and g + 8.  Tiles past the
            // matrix (last row block) hold stale stage bytes; their rows are
            // computed but never written out.
            uint32_t wv[GP][TPW][8];
            float2 sp[GP][TPW];
            uint32_t nz[GP][TPW][2];
#pragma unroll
            for (int gp = 0; gp < GP; ++gp)
#pragma unroll
                for (int r = 0; r < TPW; ++r) {
                    const uint8_t *tile = stage + ((warp * TPW + r) * W + gi0 + gp) * TBY;
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane);
                    uint32_t zp;
                    tile_meta<CMP>(tile, gq, sp[gp][r], zp);
                    nz[gp][r][0] = NEG | ((zp & 0xFFu) * 0x00010001u);
                    nz[gp][r][1] = NEG | ((zp >> 8) * 0x00010001u);
                    wv[gp][r][0] = c0.x; wv[gp][r][1] = c0.y; wv[gp][r][2] = c0.z; wv[gp][r][3] = c0.w;
                    wv[gp][r][4] = c1.x; wv[gp][r][5] = c1.y; wv[gp][r][6] = c1.z; wv[gp][r][7] = c1.w;
                }
            // k-step outer, groups and tiles inner: GP * TPW * NT independent
            // accumulator chains (a second chain per tile, even and odd
            // k-steps apart, measured 1% slower).  The A operand is q - zero
            // itself (offset + q from one LOP3, minus offset + zero by one
            // packed FMA: exact), so the MMA yields sum (q - zero) x directly
            // and a group costs one multiply by its scale.
            float d[GP][TPW][NT][4];
#pragma unroll
            for (int gp = 0; gp < GP; ++gp)
#pragma unroll
                for (int r = 0; r < TPW; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) d[gp][r][n][e] = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int gp = 0; gp < GP; ++gp) {
#pragma unroll
                    for (int r = 0; r < TPW; ++r) {
                        const uint32_t w = wv[gp][r][j];
                        const uint32_t a0 = sub_pair<ABT != 0>(lop3_and_or(w, 0x000F000Fu, MAG), nz[gp][r][0]);
                        const uint32_t a1 = sub_pair<ABT != 0>(lop3_and_or(w >> 4, 0x000F000Fu, MAG), nz[gp][r][1]);
                        const uint32_t a3 = sub_pair<ABT != 0>(lop3_and_or(w >> 8, 0x000F000Fu, MAG), nz[gp][r][1]);
                        const uint32_t a2 = sub_pair<ABT != 0>(lop3_and_or(w >> 12, 0x000F000Fu, MAG), nz[gp][r][0]);
#pragma unroll
                        for (int n = 0; n < NT; ++n)
                            mma_ab<ABT>(d[gp][r][n], a0, a1, a2, a3, bf[gp][n][j][0], bf[gp][n][j][1]);
                    }
                }
            }
#pragma unroll
            for (int gp = 0; gp < GP; ++gp) {
                if (s * W + gi0 + gp >= NG) break;  // past K: nothing to add
#pragma unroll
                for (int r = 0; r < TPW; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        float *ya = yacc[r][n];
                        ya[0] = fmaf(sp[gp][r].x, d[gp][r][n][0], ya[0]);
                        ya[1] = fmaf(sp[gp][r].x, d[gp][r][n][1], ya[1]);
                        ya[2] = fmaf(sp[gp][r].y, d[gp][r][n][2], ya[2]);
                        ya[3] = fmaf(sp[gp][r].y, d[gp][r][n][3], ya[3]);
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        if (!(it == end - 1 || s == NS - 1)) continue;

        // ----------------------------- this CTA's share of row block rb is done
        // The hand-off buffer is free once the epilogue warp has finished the
        // previous row block; the barrier makes the decision uniform.
        const bool stuck = nepi > 0 && !mbar_wait_bounded(ofree, (nepi - 1) & 1, abort_flag,
                                                          a.wait_ns, a.err);
        if (named_barrier_or(1, CONSUMERS, stuck)) return;
#pragma unroll
        for (int r = 0; r < TPW; ++r)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = (warp * TPW + r) * 16 + gq + ((e & 2) ? 8 : 0);
                    const int m = 8 * n + 2 * t + (e & 1);
                    if (m < M) out[m * (RB * 16) + row] = yacc[r][n][e];  // [m][RB * 16 rows]
                }
        named_barrier_sync(1, CONSUMERS);  // out complete before the arrival publishes it
        if (threadIdx.x == 0) mbar_arrive(ofull);
        ++nepi;
    }
}

// ABT: 0 = bf16 operands (magic 128 + q), 1 = f16 operands (magic 1024 + q).
// XSPLIT: f32 activations carried as bf16 hi + bf16 lo (two MMAs per step).
// ONE: M = 1 known at compile time (unused MMA columns skipped).
// RBT: row tiles per row block.
// CMP: compact tiles (binary16 scales, 4-bit zeros; tensor-core path only).
// ROWS: row-split consumers (2 <= M <= 16, 16-bit activations staged).
template <int MODE, int NT, int ABT, bool XSPLIT, int NSTG, bool ONE, int RBT, bool CMP, bool ROWS>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS) k_gemv(const GemvArgs a)
{
    constexpr int RB = RBT;
    constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    static_assert(!(CMP && MODE == PATH_FMA), "compact tiles: tensor-core path only");
    static_assert(!ROWS || (MODE == PATH_MMA && !XSPLIT && !ONE && RBT % W == 0), "row split");
    constexpr int TILES_BYTES = RBT * W * TBY;
    // full[NSTG], empty[NSTG], ofull, ofree, the abort flag: inside CTRL_BYTES
    static_assert((2 * NSTG + 2) * 8 + 4 <= CTRL_BYTES, "ring barriers exceed the control block");
    constexpr bool XSTAGED = (MODE == PATH_MMA) && (NT == 1 || ROWS) && !XSPLIT;
    // XS32: M = 1 f32 activations staged as f32 with the tiles (split into
    // bf16 hi + lo per step); the FMA path stages the same way
    constexpr bool XS32 = (MODE == PATH_MMA) && XSPLIT && ONE;
    const int xrows = XSTAGED ? (ONE ? 1 : a.M) : 0;
    const int SB = stage_bytes(XS32 ? PATH_FMA : MODE, xrows, RBT, TBY);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NSTG * SB);
    uint64_t *empty = full + NSTG;
    uint64_t *ofull = empty + NSTG;  // hand-off buffer written by the consumers
    uint64_t *ofree = ofull + 1;       // hand-off buffer drained by the epilogue warp
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ofree + 1);
    float *after = reinterpret_cast<float *>(smem + NSTG * SB + CTRL_BYTES);
    float *red = (MODE == PATH_FMA) ? after + W * WARP_PAIR_FLOATS : after;
    const int MSR = (MODE == PATH_FMA || ONE) ? 1 : a.M;  // red row stride
    float *out = red + (ROWS ? 0 : W * RB * 16 * MSR);  // [M][RB * 16 rows], 16-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NG = a.K / G;
    const int NS = (NG + W - 1) / W;
    const int ntiles = (a.N + TILE_ROWS - 1) / TILE_ROWS;
    const int nrb = (ntiles + RB - 1) / RB;
    const int64_t T = static_cast<int64_t>(nrb) * NS;
    const int64_t Gc = gridDim.x;
    const int64_t beg = range_begin(blockIdx.x, T, Gc);
    const int64_t end = range_begin(blockIdx.x + 1, T, Gc);
    const int xb = (a.xt == Q4_F32) ? 4 : 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTG; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);
        }
        mbar_init(ofull, 1);
        mbar_init(ofree, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // The next GEMV on the stream may begin launching; its CTAs take SMs as
    // ours exit and start streaming their (static) weights early.
    grid_dep_launch_dependents();

    // ------------------------------------------------------------ producer
    if (warp == W) {
        if (lane == 0) {
            int gstep = 0;
            if (!a.debug_no_copy) {
                // Weight tiles never depend on the previous kernel, so the
                // first NSTG stages' tiles are requested before waiting for
                // it; their activation copies follow the wait.
                auto issue_x = [&](int slot, int g0, int ng) {
                    uint8_t *stage = ring + slot * SB;
                    if (MODE == PATH_FMA || XS32)
                        bulk_g2s(stage + TILES_BYTES,
                                 static_cast<const uint8_t *>(a.x) + static_cast<int64_t>(g0) * G * xb,
                                 static_cast<uint32_t>(ng) * G * xb, &full[slot]);
                    for (int m = 0; m < xrows; ++m)
                        bulk_g2s(stage + TILES_BYTES + m * XROW,
                                 static_cast<const uint8_t *>(a.x) +
                                     (static_cast<int64_t>(m) * a.K + static_cast<int64_t>(g0) * G) * 2,
                                 static_cast<uint32_t>(ng) * G * 2, &full[slot]);
                };
                int pro_g0[NSTG], pro_ng[NSTG];
                const int npro = static_cast<int>(end - beg < NSTG ? end - beg : NSTG);
                int rb = static_cast<int>(beg / NS), s = static_cast<int>(beg % NS);
                for (int64_t it = beg; it < end; ++it, ++gstep, ++s) {
                    if (s == NS) {
                        s = 0;
                        ++rb;
                    }
                    const int slot = gstep % NSTG;
                    if (gstep >= NSTG &&
                        !mbar_wait_bounded(&empty[slot], ((gstep / NSTG) - 1) & 1, abort_flag,
                                           a.wait_ns, a.err))
                        break;
                    const int rt0 = rb * RB, nrt = min(RB, ntiles - rt0);
                    const int g0 = s * W, ng = min(W, NG - g0);
                    const uint32_t row_bytes = static_cast<uint32_t>(ng) * TBY;
                    const uint32_t xbytes = (MODE == PATH_FMA || XS32) ? static_cast<uint32_t>(ng) * G * xb
                                            : static_cast<uint32_t>(xrows) * ng * G * 2;
                    uint8_t *stage = ring + slot * SB;
                    mbar_arrive_expect_tx(&full[slot], row_bytes * nrt + xbytes);
                    // the step's tiles are contiguous in the weight buffer,
                    // row tile by row tile: one copy for a full step, one
                    // per row tile (to the stage's 4-group stride) otherwise
                    const uint8_t *src = a.qw + tile_index(rt0, g0, ntiles, NG) * TBY;
                    if (ng == W)
                        bulk_g2s(stage, src, row_bytes * nrt, &full[slot]);
                    else
                        for (int r = 0; r < nrt; ++r)
                            bulk_g2s(stage + r * W * TBY, src + r * row_bytes, row_bytes, &full[slot]);
                    if (gstep < npro) {
                        pro_g0[gstep] = g0;
                        pro_ng[gstep] = ng;
                        if (gstep == npro - 1) {
                            grid_dep_wait();
                            for (int p = 0; p < npro; ++p) issue_x(p, pro_g0[p], pro_ng[p]);
                        }
                    } else {
                        issue_x(slot, g0, ng);
                    }
                }
            }
            // Every issued copy must land before the CTA may exit.
            for (int s = max(0, gstep - NSTG); s < gstep; ++s)
                mbar_wait_bounded(&full[s % NSTG], (s / NSTG) & 1, abort_flag, a.wait_ns,
                                  a.err, false);
        }
        return;
    }

    // ------------------------------------------------------------ epilogue
    // One hand-off per row block this CTA touches, in order; the hand-off
    // buffer holds it batch row by batch row, [m][RB * 16 rows], so stores
    // to y are coalesced along the rows.  A row block held by this CTA alone
    // is written out directly.  Otherwise the partial sums go to this CTA's
    // slot of the workspace (16-byte copies) and the arrival counter is
    // stepped; the contributor that arrives last sums the partials of all
    // contributors in CTA order (the same order whoever arrives last; up to
    // eight 16-byte loads per contributor in flight per lane), and clears the
    // partials it read and the counter, so a completed call leaves the
    // workspace zero for the next one, whatever its shape.
    if (warp == W + 1) {
        // outputs and the workspace may belong to the previous kernel
        grid_dep_wait();
        if (beg < end) {
            constexpr int R16 = RB * 16;
            // one batch row (compile time): scalar partial sums, as measured
            // fastest there; otherwise 16-byte accesses
            constexpr bool M1 = MODE == PATH_FMA || ONE;
            const int Mo = M1 ? 1 : a.M;
            const int64_t slab4 = static_cast<int64_t>(R16 / 4) * Mo;  // one partial, in float4
            const int64_t slab = static_cast<int64_t>(R16) * Mo;
            const int rb_first = static_cast<int>(beg / NS), rb_last = static_cast<int>((end - 1) / NS);
            for (int rb = rb_first, e = 0; rb <= rb_last; ++rb, ++e) {
                const bool ok = mbar_wait_bounded(ofull, e & 1, abort_flag, a.wait_ns, a.err);
                if (!__all_sync(0xffffffffu, ok)) break;  // the warp leaves together
                const int64_t first_item = static_cast<int64_t>(rb) * NS;
                const int c_first = static_cast<int>(owner_of(first_item, T, Gc));
                const int c_last = static_cast<int>(owner_of(first_item + NS - 1, T, Gc));
                const int nc = c_last - c_first + 1;
                const int row0 = rb * R16;
                const int nout = min(RB, ntiles - rb * RB) * 16 * Mo;
                const int nval = min(min(RB, ntiles - rb * RB) * 16, a.N - row0);  // rows that exist
                if (nc == 1) {
                    if constexpr (M1) {
                        for (int i = lane; i < nout; i += 32)
                            if (row0 + i < a.N) put_y(a, row0 + i, out[i]);
                    } else {
                        for (int i = lane; i < Mo * R16; i += 32) {
                            const int m = i / R16, row = i % R16;
                            if (row < nval)
                                put_y(a, static_cast<int64_t>(m) * a.N + row0 + row, out[i]);
                        }
                    }
                } else if constexpr (M1) {
                    float *part = a.partial + (static_cast<int64_t>(rb) * a.maxc) * slab;
                    for (int i = lane; i < nout; i += 32)
                        put_part(a, &part[(blockIdx.x - c_first) * slab + i], out[i]);
                    __syncwarp();
                    unsigned int prev = 0;
                    if (lane == 0 && count_ok(a, rb)) prev = atomic_add_acq_rel_gpu(&a.count[rb], 1u);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    __syncwarp();
                    if (prev == static_cast<unsigned int>(nc - 1)) {
                        // last to arrive: every partial is visible.  Four
                        // outputs x four contributors of loads in flight at
                        // once; the sums still run in CTA order.
                        for (int i0 = lane; i0 < nout; i0 += 4 * 32) {
                            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            for (int c0 = 0; c0 < nc; c0 += 4) {
                                float pv[4][4];
#pragma unroll
                                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        const int i = i0 + 32 * u;
                                        pv[cc][u] = (c0 + cc < nc && i < nout)
                                                        ? __ldcg(&part[(c0 + cc) * slab + i])
                                                        : 0.0f;
                                    }
#pragma unroll
                                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                                    for (int u = 0; u < 4; ++u)
                                        if (c0 + cc < nc) {
                                            v[u] += pv[cc][u];
                                            // consumed: the workspace goes back to zero
                                            if (i0 + 32 * u < nout)
                                                put_part(a, &part[(c0 + cc) * slab + i0 + 32 * u], 0.0f);
                                        }
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = i0 + 32 * u;
                                if (i >= nout) continue;
                                const int row = i / Mo, m = i % Mo;
                                if (row0 + row < a.N)
                                    put_y(a, static_cast<int64_t>(m) * a.N + row0 + row, v[u]);
                            }
                        }
                        if (lane == 0 && count_ok(a, rb)) a.count[rb] = 0u;  // ready for the next call
                    }
                } else {
                    float4 *part = reinterpret_cast<float4 *>(a.partial) + (static_cast<int64_t>(rb) * a.maxc) * slab4;
                    float4 *mine = part + (blockIdx.x - c_first) * slab4;
                    const float4 *o4 = reinterpret_cast<const float4 *>(out);
                    for (int i = lane; i < slab4; i += 32) put_part4(a, &mine[i], o4[i]);
                    __syncwarp();
                    unsigned int prev = 0;
                    if (lane == 0 && count_ok(a, rb)) prev = atomic_add_acq_rel_gpu(&a.count[rb], 1u);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    __syncwarp();
                    if (prev == static_cast<unsigned int>(nc - 1)) {
                        // last to arrive: every partial is visible.  U
                        // 16-byte loads per lane for each of two contributors
                        // in flight at once (8 for the larger partials of two
                        // batch tiles; 4 measured faster below); the sums run
                        // in CTA order.
                        constexpr int U = NT == 2 ? 8 : 4;
                        for (int i0 = lane; i0 < slab4; i0 += U * 32) {
                            float4 v[U];
#pragma unroll
                            for (int u = 0; u < U; ++u) v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int c0 = 0; c0 < nc; c0 += 2) {
                                float4 pv[2][U];
#pragma unroll
                                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                                    for (int u = 0; u < U; ++u) {
                                        const int64_t i = i0 + 32 * u;
                                        pv[cc][u] = (c0 + cc < nc && i < slab4)
                                                        ? __ldcg(&part[(c0 + cc) * slab4 + i])
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                                    }
#pragma unroll
                                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                                    for (int u = 0; u < U; ++u) {
                                        const int64_t i = i0 + 32 * u;
                                        if (c0 + cc < nc && i < slab4) {
                                            v[u].x += pv[cc][u].x;
                                            v[u].y += pv[cc][u].y;
                                            v[u].z += pv[cc][u].z;
                                            v[u].w += pv[cc][u].w;
                                            // consumed: the workspace goes back to zero
                                            put_part4(a, &part[(c0 + cc) * slab4 + i],
                                                      make_float4(0.f, 0.f, 0.f, 0.f));
                                        }
                                    }
                            }
#pragma unroll
                            for (int u = 0; u < U; ++u) {
                                const int i = i0 + 32 * u;
                                if (i >= slab4) continue;
                                const int m = (4 * i) / R16, row = (4 * i) % R16;
                                const int64_t yb = static_cast<int64_t>(m) * a.N + row0 + row;
                                if (row < nval) put_y(a, yb, v[u].x);
                                if (row + 1 < nval) put_y(a, yb + 1, v[u].y);
                                if (row + 2 < nval) put_y(a, yb + 2, v[u].z);
                                if (row + 3 < nval) put_y(a, yb + 3, v[u].w);
                            }
                        }
                        if (lane == 0 && count_ok(a, rb)) a.count[rb] = 0u;  // ready for the next call
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ofree);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    // Activations may belong to the previous kernel on the stream: touch
    // them only after it has completed.
    grid_dep_wait();
    if constexpr (ROWS) {
        consume_rows<NT, ABT, NSTG, RBT, CMP>(a, ring, SB, full, empty, ofull, ofree, abort_flag,
                                               out, beg, end, NS, ntiles, NG);
    } else {
    const int gq = lane >> 2, t = lane & 3;
    const int M = ONE ? 1 : a.M;
    const int MS = MSR;
    const int Mo = (MODE == PATH_FMA) ? 1 : M;
    float *mypairs = after + warp * WARP_PAIR_FLOATS;  // FMA

    // MMA: the warp's B fragments for the current step, the next step's
    // prefetched while the current one computes (f32 hi/lo: loaded per step)
    constexpr bool PREFETCH = (MODE == PATH_MMA) && !XSPLIT && !XSTAGED;
    uint32_t bcur[NT][8][2], bnxt[PREFETCH ? NT : 1][8][2], blo[XSPLIT ? NT : 1][8][2];
    auto load_b = [&](int gg, uint32_t (&bh)[NT][8][2], uint32_t (&bl)[XSPLIT ? NT : 1][8][2]) {
        const bool act = gg < NG;
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
    if (MODE == PATH_MMA && !XSTAGED && !XS32 && beg < end)
        load_b(static_cast<int>(beg % NS) * W + warp, bcur, blo);

    float yacc[RB][NT][4];
    int gstep = 0, nepi = 0;
    bool ok = true;
    int rb = static_cast<int>(beg / NS), s = static_cast<int>(beg % NS) - 1;
    for (int64_t it = beg; it < end; ++it, ++gstep) {
        if (++s == NS) {
            s = 0;
            ++rb;
        }
        const int slot = gstep % NSTG;
        const int g = s * W + warp;
        const bool active = g < NG;
        const int nrt = min(RB, ntiles - rb * RB);
        if (it == beg || s == 0) {
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) yacc[r][n][e] = 0.0f;
        }

        ok = mbar_wait_bounded(&full[slot], (gstep / NSTG) & 1, abort_flag, a.wait_ns, a.err);
        if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
        }
        if (MODE == PATH_MMA && XSPLIT && !XS32 && it > beg) load_b(g, bcur, blo);
        if (PREFETCH && it + 1 < end)
            load_b((s + 1 == NS ? 0 : s + 1) * W + warp,
                   reinterpret_cast<uint32_t (&)[NT][8][2]>(bnxt), blo);
        const uint8_t *stage = ring + slot * SB;
        const uint8_t *wtiles = stage + warp * TBY;
        if (XS32) {
            // B fragments (k = 16j + 2t + {0, 1} and + 8) of the single
            // activation row, each f32 pair split into bf16 hi + bf16 lo
            const float *xs = reinterpret_cast<const float *>(stage + TILES_BYTES) + warp * G + 2 * t;
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 xv = *reinterpret_cast<const float2 *>(xs + 16 * j + 8 * h);
                    const uint32_t vh = pack_bf16x2(xv.x, xv.y);
                    bcur[0][j][h] = vh;
                    blo[0][j][h] = pack_bf16x2(xv.x - bf16_lo_f32(vh), xv.y - bf16_hi_f32(vh));
                }
        }
        if (XSTAGED) {
            // Lanes of batch rows >= M read row M - 1: their MMA columns are
            // never stored, and an MMA column depends on its own B column
            // only.  An idle warp's reads stay inside the stage too.
            const int xr = gq < M ? gq : M - 1;
            const uint8_t *xs = stage + TILES_BYTES + xr * XROW + warp * G * 2 + 4 * t;
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    bcur[0][j][h] = *reinterpret_cast<const uint32_t *>(xs + 32 * j + 16 * h);
        }

        if (active && MODE == PATH_FMA) {
            // This warp's group activations -> pair records.  Lane (tt, j)
            // writes word j of lane class tt: (x1,x8) (x9,x1) (x8,x0)
            // (x0',x9) with xa = x[16j + 2tt + a] and x0' from the next word
            // of the same 16-byte chunk (see the word layout in q4.h).
            {
                const int tt = lane >> 3, j = lane & 7;
                const int jn = (j & 4) | ((j + 1) & 3);
                const uint8_t *xs = stage + TILES_BYTES;
                const int kb = warp * G + 2 * tt;
                const float x0 = smem_x_f32(xs, a.xt, kb + 16 * j);
                const float x1 = smem_x_f32(xs, a.xt, kb + 16 * j + 1);
                const float x8 = smem_x_f32(xs, a.xt, kb + 16 * j + 8);
                const float x9 = smem_x_f32(xs, a.xt, kb + 16 * j + 9);
                const float x0n = smem_x_f32(xs, a.xt, kb + 16 * jn);
                float4 *dst = reinterpret_cast<float4 *>(mypairs + tt * PAIR_STRIDE + 8 * j);
                dst[0] = make_float4(x1, x8, x9, x1);
                dst[1] = make_float4(x8, x0, x0n, x9);
                float slo = x0 + x1, shi = x8 + x9;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    slo += __shfl_xor_sync(0xffffffffu, slo, o);
                    shi += __shfl_xor_sync(0xffffffffu, shi, o);
                }
                if (j == 0)
                    reinterpret_cast<float4 *>(mypairs + 4 * PAIR_STRIDE)[tt] =
                        make_float4(slo + shi, 128.0f * slo + 2048.0f * shi,
                                    128.0f * shi + 2048.0f * slo, 0.0f);
            }
            __syncwarp();
            const float4 *xpp = reinterpret_cast<const float4 *>(mypairs + t * PAIR_STRIDE);
            float2 P[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 p = xpp[2 * j], q = xpp[2 * j + 1];
                P[j][0] = make_float2(p.x, p.y);
                P[j][1] = make_float2(p.z, p.w);
                P[j][2] = make_float2(q.x, q.y);
                P[j][3] = make_float2(q.z, q.w);
            }
            const float4 xsv = reinterpret_cast<const float4 *>(mypairs + 4 * PAIR_STRIDE)[t];
            // all RB tiles at once: RB independent accumulator chains
            uint32_t wv[RB][8];
            float2 sp[RB];
            uint32_t zp[RB];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const uint8_t *tile = wtiles + r * W * TBY;
                const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane);
                sp[r] = *reinterpret_cast<const float2 *>(tile + SCALE_OFF + 8 * gq);
                zp[r] = *reinterpret_cast<const uint16_t *>(tile + ZERO_OFF + 2 * gq);
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
                    fma_word(accG[r], accG8[r], wv[r][j], wv[r][(j & 4) | ((j + 1) & 3)], P[j][0],
                             P[j][1], P[j][2], P[j][3]);
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
            // TI tiles at a time: TI * NT independent accumulator chains, plus
            // NT chains for the activation sums
            constexpr int TI0 = (NT == 1) ? 4 : 2;
            constexpr int TI = TI0 < RB ? TI0 : RB;
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
                    const uint8_t *tile = wtiles + (r0 + i) * W * TBY;
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(tile + 16 * lane);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(tile + 512 + 16 * lane);
                    tile_meta<CMP>(tile, gq, sp[i], zp[i]);
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
                        if (NT == 1 && !XSPLIT) {
                            mma_word<ABT>(d[i][0], w, bcur[0][j][0], bcur[0][j][1]);
                        } else {
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
                }
#pragma unroll
                for (int i = 0; i < TI; ++i) {
                    // OFF + zero: the byte under the exponent of 2^23, one
                    // permute and one add each
                    const float zg = __uint_as_float(__byte_perm(zp[i], 0x4B000000u, 0x7540)) -
                                     (8388608.0f - OFF);
                    const float zg8 = __uint_as_float(__byte_perm(zp[i], 0x4B000000u, 0x7541)) -
                                      (8388608.0f - OFF);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        float *ya = yacc[r0 + i][n];
                        ya[0] = fmaf(sp[i].x, fmaf(-zg, S[n][0], d[i][n][0]), ya[0]);
                        ya[2] = fmaf(sp[i].y, fmaf(-zg8, S[n][0], d[i][n][2]), ya[2]);
                        if (!ONE) {  // second MMA column: batch rows 2t + 1
                            ya[1] = fmaf(sp[i].x, fmaf(-zg, S[n][1], d[i][n][1]), ya[1]);
                            ya[3] = fmaf(sp[i].y, fmaf(-zg8, S[n][1], d[i][n][3]), ya[3]);
                        }
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

        if (!(it == end - 1 || s == NS - 1)) continue;

        // ----------------------------- this CTA's share of row block rb is done
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
                        if (m < M) red[(warp * RB * 16 + row) * MS + m] = yacc[r][n][e];
                    }
        }
        // The hand-off buffer is free once the epilogue warp has finished
        // the previous row block; the barrier makes the decision uniform.
        const bool stuck = nepi > 0 && !mbar_wait_bounded(ofree, (nepi - 1) & 1, abort_flag,
                                                          a.wait_ns, a.err);
        if (named_barrier_or(1, CONSUMERS, stuck)) {
            ok = false;
            break;
        }
        if constexpr (MODE == PATH_FMA || ONE) {  // one batch row: [rows]
            for (int i = threadIdx.x; i < nrt * 16; i += CONSUMERS) {
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < W; ++w) v += red[w * RB * 16 + i];
                out[i] = v;
            }
        } else {
            const int nrows = nrt * 16;
            for (int i = threadIdx.x; i < nrows * Mo; i += CONSUMERS) {
                const int m = i / nrows, row = i % nrows;
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < W; ++w) v += red[(w * RB * 16 + row) * MS + m];
                out[m * (RB * 16) + row] = v;  // hand-off layout [m][RB * 16 rows]
            }
        }
        // red is reused by the next row block; the arrival publishes out
        named_barrier_sync(1, CONSUMERS);
        if (threadIdx.x == 0) mbar_arrive(ofull);
        ++nepi;
    }
    }  // !ROWS
}

// -------------------------------------------------------------------- host
template <int MODE, int NT, int ABT, bool XSPLIT, int NSTG = NSTAGE, bool ONE = false, int RBT = RB,
          bool CMP = false, bool ROWS = false>
struct Kern {
    static constexpr bool XSTAGED = (MODE == PATH_MMA) && (NT == 1 || ROWS) && !XSPLIT;
    static constexpr bool XS32 = (MODE == PATH_MMA) && XSPLIT && ONE;
    static constexpr int TBY = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    static int smem(int M)
    {
        if (XS32)  // f32 staging as in the FMA path, MMA-sized reduction buffers
            return NSTG * stage_bytes(PATH_FMA, 0, RBT, TBY) + CTRL_BYTES + W * RBT * 16 * 4 +
                   RBT * 16 * 4;
        if (ROWS)  // staged rows, no cross-warp reduction buffer
            return NSTG * stage_bytes(MODE, M, RBT, TBY) + CTRL_BYTES + RBT * 16 * M * 4;
        return smem_bytes(MODE, XSTAGED ? M : 0, MODE == PATH_FMA ? 1 : M, NSTG, RBT, TBY);
    }
    static cudaError_t configure(int dev, int M, int *blocks_per_sm)
    {
        // per-device caches; concurrent first calls may both fill them (the
        // same values), so relaxed atomics suffice
        static std::atomic<int> cached[64][17];
        static std::atomic<bool> attr[64];
        if (dev < 0 || dev >= 64 || M < 1 || M > 16) return cudaErrorInvalidValue;
        const int known = cached[dev][M].load(std::memory_order_relaxed);
        if (known > 0) {
            *blocks_per_sm = known;
            return cudaSuccess;
        }
        auto kern = k_gemv<MODE, NT, ABT, XSPLIT, NSTG, ONE, RBT, CMP, ROWS>;
        if (!attr[dev].load(std::memory_order_relaxed)) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 smem(NSTG == NSTAGE ? 16 : 1));
            if (e != cudaSuccess) return e;
            attr[dev].store(true, std::memory_order_relaxed);
        }
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, THREADS, smem(M));
        if (e != cudaSuccess) return e;
        if (n < 1) n = 1;
        cached[dev][M].store(n, std::memory_order_relaxed);
        *blocks_per_sm = n;
        return cudaSuccess;
    }
    static cudaError_t launch(int grid, const GemvArgs &a, cudaStream_t s)
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem(a.M);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, k_gemv<MODE, NT, ABT, XSPLIT, NSTG, ONE, RBT, CMP, ROWS>, a);
    }
};

template <bool CMP, typename F>
static cudaError_t dispatch_t(int path, int M, q4_dtype xt, bool deep, bool small, F &&f)
{
    if (path == PATH_FMA) {
        if constexpr (CMP) return cudaErrorInvalidValue;  // rejected before planning
        else return f(Kern<PATH_FMA, 1, 0, false>{});
    }
    // 2 <= M <= 8, 16-bit activations: group-split consumers, one MMA
    // column tile for the batch rows, the step's activation rows staged
    if (M >= 2 && M <= 8 && xt != Q4_F32) {
        if (xt == Q4_F16) return f(Kern<PATH_MMA, 1, 1, false, NSTAGE, false, RB, CMP>{});
        return f(Kern<PATH_MMA, 1, 0, false, NSTAGE, false, RB, CMP>{});
    }
    // 9 <= M <= 16, 16-bit activations: row-split consumers, two MMA column
    // tiles (4-tile row blocks for small problems)
    if (M >= 9 && xt != Q4_F32) {
        if (small) {
            if (xt == Q4_F16) return f(Kern<PATH_MMA, 2, 1, false, NSTAGE, false, RB_SMALL_ROWS, CMP, true>{});
            return f(Kern<PATH_MMA, 2, 0, false, NSTAGE, false, RB_SMALL_ROWS, CMP, true>{});
        }
        if (xt == Q4_F16) return f(Kern<PATH_MMA, 2, 1, false, NSTAGE, false, RB, CMP, true>{});
        return f(Kern<PATH_MMA, 2, 0, false, NSTAGE, false, RB, CMP, true>{});
    }
    // deep: M = 1, where a 3-stage ring still fits two CTAs per SM
    const bool two = M > 8;
    if (xt == Q4_F16)  // M == 1
        return deep ? f(Kern<PATH_MMA, 1, 1, false, 3, true, RB, CMP>{})
                    : f(Kern<PATH_MMA, 1, 1, false, NSTAGE, true, RB, CMP>{});
    if (xt == Q4_BF16)
        return deep ? f(Kern<PATH_MMA, 1, 0, false, 3, true, RB, CMP>{})
                    : f(Kern<PATH_MMA, 1, 0, false, NSTAGE, true, RB, CMP>{});
    if (M == 1)
        return deep ? f(Kern<PATH_MMA, 1, 0, true, 3, true, RB, CMP>{})
                    : f(Kern<PATH_MMA, 1, 0, true, NSTAGE, true, RB, CMP>{});
    return two ? f(Kern<PATH_MMA, 2, 0, true, NSTAGE, false, RB, CMP>{})
               : f(Kern<PATH_MMA, 1, 0, true, NSTAGE, false, RB, CMP>{});
}

// cmp: compact tiles (binary16 scales, 4-bit zeros)
template <typename F>
static cudaError_t dispatch(bool cmp, int path, int M, q4_dtype xt, bool deep, bool small, F &&f)
{
    return cmp ? dispatch_t<true>(path, M, xt, deep, small, f)
               : dispatch_t<false>(path, M, xt, deep, small, f);
}

size_t gemv_counter_bytes(int64_t N)
{
    return ((static_cast<size_t>((N + 31) / 32) * sizeof(unsigned int) + 255) / 256) * 256;
}

static GemvPlan make_plan(int M, int N, int K, q4_dtype xt, int path, int sm_count, bool cmp);

// Plans depend only on (device, shape, activation type, path, tile layout);
// a decode loop asks for the same few again and again, so they are kept (a
// small map, cleared if it ever grows large).
GemvPlan gemv_plan(int M, int N, int K, q4_dtype xt, int path, int sm_count, bool cmp)
{
    struct Key {
        int dev, M, N, K, xt, path, sms, cmp;
        bool operator==(const Key &o) const
        {
            return dev == o.dev && M == o.M && N == o.N && K == o.K && xt == o.xt &&
                   path == o.path && sms == o.sms && cmp == o.cmp;
        }
    };
    struct Hash {
        size_t operator()(const Key &k) const
        {
            uint64_t h = 1469598103934665603ull;
            for (int v : {k.dev, k.M, k.N, k.K, k.xt, k.path, k.sms, k.cmp})
                h = (h ^ static_cast<uint32_t>(v)) * 1099511628211ull;
            return static_cast<size_t>(h);
        }
    };
    static std::mutex mu;
    static std::unordered_map<Key, GemvPlan, Hash> plans;
    int dev = 0;
    cudaGetDevice(&dev);
    const Key key{dev, M, N, K, static_cast<int>(xt), path, sm_count, cmp ? 1 : 0};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = plans.find(key);
        if (it != plans.end()) return it->second;
    }
    const GemvPlan p = make_plan(M, N, K, xt, path, sm_count, cmp);
    if (p.grid > 0) {  // a plan whose kernel configuration failed is not kept
        std::lock_guard<std::mutex> lock(mu);
        if (plans.size() > 4096) plans.clear();
        plans.emplace(key, p);
    }
    return p;
}

static GemvPlan make_plan(int M, int N, int K, q4_dtype xt, int path, int sm_count, bool cmp)
{
    GemvPlan p{};
    p.cmp = cmp;
    // AUTO: the tensor-core path (its unpack costs 7 ALU instructions per 8
    // weights against 11 for the CUDA-core path, which is bound by the ALU
    // pipe); f32 activations ride as bf16 hi + lo with two MMAs per word,
    // staged as f32 with the tiles at M = 1 (measured 6-11% faster than the
    // CUDA-core path there).
    if (path == PATH_AUTO) path = PATH_MMA;
    p.path = path;
    const int ntiles = (N + TILE_ROWS - 1) / TILE_ROWS;
    const int NG = K / G;
    const int NS = (NG + W - 1) / W;
    int dev = 0, per_sm = 1;
    cudaGetDevice(&dev);
    cudaError_t cfg = dispatch(cmp, path, M, xt, false, false,
                               [&](auto k) { return decltype(k)::configure(dev, M, &per_sm); });
    // Fewer than 8 steps per CTA with 8-tile row blocks, 9 <= M <= 16 (the
    // row-split consumers): use 4-tile ones (one row tile per consumer
    // warp), so that steps are short and plentiful (the 70B decode step at
    // M = 16: 2.4% faster than below 4 steps; the group-split consumers of
    // M <= 8 keep 8-tile blocks).
    const int64_t T8 = static_cast<int64_t>((ntiles + RB - 1) / RB) * NS;
    p.small = T8 < 8 * static_cast<int64_t>(sm_count) * per_sm && path == PATH_MMA && M >= 9 &&
              xt != Q4_F32;
    if (p.small && cfg == cudaSuccess)
        cfg = dispatch(cmp, path, M, xt, false, true,
                       [&](auto k) { return decltype(k)::configure(dev, M, &per_sm); });
    p.rb = p.small ? RB_SMALL_ROWS : RB;
    p.nrb = (ntiles + p.rb - 1) / p.rb;
    const int64_t T = static_cast<int64_t>(p.nrb) * NS;
    const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
    p.grid = static_cast<int>(T < slots ? T : slots);
    // With few steps per CTA, give every CTA the same whole number of steps
    // (a 3-or-4 split leaves a quarter of the CTAs a step behind); measured
    // 1.5% faster on the 70B decode step.
    if (T > slots && T < 8 * slots) {
        const int64_t per = (T + slots - 1) / slots;
        p.grid = static_cast<int>((T + per - 1) / per);
    }
    // M = 1: the 3-stage ring whenever it fits (measured on the 70B decode
    // step: +0.3% against keeping the 2-stage ring for CTAs of under 5 steps).
    p.deep = !p.small && path == PATH_MMA && M == 1;
    if (p.deep) {  // same CTAs per SM, or keep the 2-stage ring
        int per_sm_deep = 0;
        dispatch(cmp, path, M, xt, true, false,
                 [&](auto k) { return decltype(k)::configure(dev, M, &per_sm_deep); });
        p.deep = per_sm_deep == per_sm;
    }
    // most CTAs sharing one row block
    int maxc = 1;
    for (int64_t rb = 0; rb < p.nrb; ++rb) {
        const int64_t c0 = owner_of(rb * NS, T, p.grid), c1 = owner_of(rb * NS + NS - 1, T, p.grid);
        if (c1 - c0 + 1 > maxc) maxc = static_cast<int>(c1 - c0 + 1);
    }
    p.maxc = maxc;
    p.workspace = maxc > 1 ? gemv_counter_bytes(N) + static_cast<size_t>(p.nrb) * maxc * p.rb * 16 *
                                                         static_cast<size_t>(M) * sizeof(float)
                           : 0;
    if (cfg != cudaSuccess) p.grid = 0;  // the launch then fails and reports it
    return p;
}

cudaError_t gemv_launch(const GemvPlan &p, const GemvArgs &a, cudaStream_t s)
{
    return dispatch(p.cmp, p.path, a.M, a.xt, p.deep, p.small,
                    [&](auto k) { return decltype(k)::launch(p.grid, a, s); });
}

}  // namespace q4
