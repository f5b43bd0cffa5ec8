// common.cuh -- shared constants, inline-PTX helpers and internal launcher
// declarations of the q4 library (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "../../include/q4.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace q4 {

constexpr int G = Q4_GROUP;                 // weights per group along K
constexpr int TILE_ROWS = Q4_TILE_ROWS;     // rows per tile
constexpr int TILE_BYTES = Q4_TILE_BYTES;   // 1104
constexpr int CODE_BYTES = 1024;            // 16 rows x 128 codes / 2
constexpr int SCALE_OFF = 1024;             // 8 pairs of f32 scales
constexpr int ZERO_OFF = 1088;              // 8 pairs of u8 zeros
// Compact tiles: the same codes, then 8 pairs of binary16 scales (bytes
// 1024..1055), 8 bytes of zero-nibble pairs (z_i | z_{i+8} << 4), 8 bytes of
// padding: 1072 = 67 x 16 bytes, so every tile stays 16-byte aligned.
constexpr int CMP_TILE_BYTES = Q4_CMP_TILE_BYTES;  // 1072
constexpr int CMP_ZERO_OFF = 1056;

// Device error word (one per device, defined in api.cu, its address passed to
// every kernel that waits): bit 0 = a bounded wait timed out.  Read and
// cleared by q4_check.
constexpr unsigned int ERR_TIMEOUT = 1u;
constexpr unsigned int ERR_BOUNDS = 2u;  // a store outside its buffer (Q4_DEBUG builds)
unsigned int *device_error_word();  // host: address on the current device

#ifdef Q4_DEBUG
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Debug builds (-DQ4_DEBUG) check every global store of the kernels against
// the extent of its buffer: an index outside [0, limit) raises ERR_BOUNDS in
// the device error word and the caller skips the store (no trap, no fault;
// q4_check reports Q4_ERR_BOUNDS).  Release builds compile the check away.
__device__ __forceinline__ bool store_ok(int64_t idx, int64_t limit, unsigned int *err)
{
    if constexpr (!kDebugBounds) return true;
    if (idx >= 0 && idx < limit) return true;
    if (err) atomicOr(err, ERR_BOUNDS);
    return false;
}

// Host: keeps the CUDA error's text for q4_last_cuda_error (this thread) and
// returns Q4_ERR_CUDA.
q4_status cuda_fail(cudaError_t e);

// Host: bytes of an N x K weight buffer in `layout` (0 if invalid).
size_t weight_bytes(int64_t N, int64_t K, q4_layout layout);

// ----------------------------------------------------------------- inline PTX
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// One potentially blocking probe of an mbarrier phase: the thread may be
// suspended in hardware (up to about 0.5 ms) until the phase completes, so
// waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
        : "memory");
    return ok != 0;
}

// One non-blocking probe of an mbarrier phase (for latency-critical waiters
// that poll instead of being suspended).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  Returns false (after raising the
// device error word and the CTA's abort flag) when `limit_ns` elapses or when
// another role of the CTA has already aborted.  Never spins without bound.
// With honor_abort == false (used to drain copies already in flight before
// a CTA exits) only the time bound ends the wait.
// With poll == true the waiter probes without being suspended (reacts
// sooner, takes issue slots meanwhile).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort_flag, uint64_t limit_ns,
                                                  unsigned int *err, bool honor_abort = true,
                                                  bool poll = false)
{
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(err, ERR_TIMEOUT);
            return false;
        }
    }
}

// 1-D bulk asynchronous copy global -> shared (TMA engine, no tensor map),
// completion counted in bytes on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads:
// every thread gets the same answer, so a decision taken on it is uniform.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Arrival counter step with acquire-release semantics at GPU scope: orders
// the caller's earlier writes (and those ordered before them by a barrier)
// before the increment, and later reads after it.
__device__ __forceinline__ unsigned int atomic_add_acq_rel_gpu(unsigned int *p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Programmatic dependent launch: let the next kernel on the stream start
// launching (its CTAs become resident as ours exit), and wait until the
// previous kernel on the stream has completed and its writes are visible.
__device__ __forceinline__ void grid_dep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// d = (a & b) | c  as one LOP3
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = a * 1 + c on a pair of 16-bit floats (bf16, or f16 when F16); exact
// where it is used: a is offset + q, c = -(offset + zero), and the difference
// q - zero is a small integer.
template <bool F16>
__device__ __forceinline__ uint32_t sub_pair(uint32_t a, uint32_t c)
{
    uint32_t d;
    if (F16)
        asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3C003C00u), "r"(c));
    else
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3F803F80u), "r"(c));
    return d;
}

// ------------------------------------------------------------ tile order
// Order of the tiles in both tiled layouts: blocks of LB_TILES row tiles
// (128 rows); inside a block, steps of LB_GROUPS groups (512 k); inside a
// step, row tile then group.  One step of one block -- the unit a decode
// GEMV consumes -- is thus one contiguous run of up to 32 tiles.  The last
// block may hold fewer row tiles and the last step fewer groups; every
// earlier block and step is full.
constexpr int LB_TILES = 8;
constexpr int LB_GROUPS = 4;

// Index (in tiles) of tile (row tile rt, group g) of a matrix of ntiles row
// tiles and NG groups.
__host__ __device__ __forceinline__ int64_t tile_index(int64_t rt, int g, int64_t ntiles, int NG)
{
    const int64_t rb = rt / LB_TILES;
    const int64_t nrt = ntiles - rb * LB_TILES < LB_TILES ? ntiles - rb * LB_TILES : LB_TILES;
    const int s = g / LB_GROUPS;
    const int ng = NG - s * LB_GROUPS < LB_GROUPS ? NG - s * LB_GROUPS : LB_GROUPS;
    return rb * LB_TILES * NG + s * nrt * LB_GROUPS + (rt - rb * LB_TILES) * ng + (g - s * LB_GROUPS);
}

// Inverse of tile_index: the (row tile, group) of the t-th tile.
__host__ __device__ __forceinline__ void tile_of(int64_t t, int64_t ntiles, int NG, int64_t &rt, int &g)
{
    const int64_t per_block = static_cast<int64_t>(LB_TILES) * NG;
    const int64_t rb = t / per_block;
    const int64_t rem = t - rb * per_block;
    const int64_t nrt = ntiles - rb * LB_TILES < LB_TILES ? ntiles - rb * LB_TILES : LB_TILES;
    const int NS = (NG + LB_GROUPS - 1) / LB_GROUPS;
    int64_t s = rem / (nrt * LB_GROUPS);
    if (s > NS - 1) s = NS - 1;
    const int64_t rem2 = rem - s * nrt * LB_GROUPS;
    const int ng = NG - static_cast<int>(s) * LB_GROUPS < LB_GROUPS ? NG - static_cast<int>(s) * LB_GROUPS
                                                                    : LB_GROUPS;
    rt = rb * LB_TILES + rem2 / ng;
    g = static_cast<int>(s) * LB_GROUPS + static_cast<int>(rem2 % ng);
}

// ------------------------------------------------------------ dtype helpers
__device__ __forceinline__ float load_x_f32(const void *x, q4_dtype xt, int64_t i)
{
    if (xt == Q4_F32) return static_cast<const float *>(x)[i];
    const uint16_t b = static_cast<const uint16_t *>(x)[i];
    if (xt == Q4_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
    __half_raw hr;
    hr.x = b;
    return __half2float(__half(hr));
}

// ------------------------------------------------------- internal launchers
struct GemvArgs {
    const void *x;
    q4_dtype xt;
    int M, N, K;
    const uint8_t *qw;
    void *y;
    q4_dtype yt;
    float *partial;       // [nrb][maxc][64 rows][M] partial sums of shared row blocks
    unsigned int *count;  // [nrb] arrival counters of shared row blocks
    int64_t partial_len;  // floats the workspace holds at `partial` (store checks)
    int64_t count_len;    // counters the workspace holds at `count` (store checks)
    int maxc;             // most CTAs that share one row block
    uint64_t wait_ns;     // bound of every mbarrier wait
    unsigned int *err;    // device error word
    int debug_no_copy;    // producer issues no copy (exercises the timeout path)
};

enum GemvPath { PATH_AUTO = 0, PATH_FMA = 1, PATH_MMA = 2 };

struct GemvPlan {
    int path;
    int rb;    // row tiles per row block
    int nrb;   // row blocks
    int grid;  // persistent CTAs
    int maxc;  // most CTAs sharing one row block (1: no partial sums)
    bool deep; // 3-stage ring (M = 1, 16-bit activations, many steps per CTA)
    bool small;  // 2-tile row blocks (few steps per CTA)
    bool cmp;    // compact tiles (binary16 scales, 4-bit zeros)
    size_t workspace;
};

GemvPlan gemv_plan(int M, int N, int K, q4_dtype xt, int path, int sm_count, bool cmp = false);
// Counter block at the start of the workspace: one u32 arrival counter per
// 32 output rows (at least one per row block), padded to 256 bytes.
size_t gemv_counter_bytes(int64_t N);
cudaError_t gemv_launch(const GemvPlan &plan, const GemvArgs &a, cudaStream_t s);

cudaError_t quantize_launch(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                            uint8_t *zero, bool symmetric, unsigned int *err, cudaStream_t s);
cudaError_t repack_launch(const uint8_t *packed, const float *scale, const uint8_t *zero,
                          int64_t N, int64_t K, uint8_t *qw, unsigned int *err, cudaStream_t s);
cudaError_t unpack_launch(const uint8_t *qw, int64_t N, int64_t K, uint8_t *packed, float *scale,
                          uint8_t *zero, unsigned int *err, cudaStream_t s);
cudaError_t repack_compact_launch(const uint8_t *packed, const float *scale, const uint8_t *zero,
                                  int64_t N, int64_t K, uint8_t *qw, unsigned int *err,
                                  cudaStream_t s);
cudaError_t unpack_compact_launch(const uint8_t *qw, int64_t N, int64_t K, uint8_t *packed,
                                  uint16_t *scale16, uint8_t *zero, unsigned int *err,
                                  cudaStream_t s);
// Large-M GEMM plan: tiles of 128 weight rows x bt tokens; either every
// tile is computed by one CTA (split == false, tiles dealt round robin) or
// the tiles' groups form one sequence of items cut into equal contiguous
// ranges, one per CTA, with partial sums through the workspace.
struct GemmPlan {
    int bt;        // tokens per tile: 16, 32, 64 or 128
    int mt, nt;    // tiles along M and along N
    int grid;      // persistent CTAs
    bool split;    // groups of a tile may be spread over several CTAs
    int maxc;      // most CTAs sharing one tile (1 without split)
    size_t workspace;
};
GemmPlan gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count);
q4_status gemm_run(const GemmPlan &p, const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                   const uint8_t *qw, bool cmp, void *y, q4_dtype yt, void *workspace,
                   unsigned int *err, uint64_t wait_ns, int debug_no_copy, cudaStream_t s,
                   cudaError_t *cerr);
cudaError_t xsum_launch(const void *x, q4_dtype xt, int64_t M, int64_t K, float *xsum,
                        unsigned int *err, cudaStream_t s);

}  // namespace q4
