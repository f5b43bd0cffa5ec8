/*
 * q4.h -- C ABI of the GB300 (sm_103a) weight-only INT4 group-128 library.
 *
 * What is computed (page "Weight quantization", tirogla.com, section "How it
 * works" and section "Code"):
 *   for each group of G = 128 consecutive weights of a row, along the input
 *   dimension K:
 *     lo = min(min w, 0), hi = max(max w, 0)
 *     scale = (hi - lo) / 15            (1 when hi == lo)
 *     zero  = clamp(round(-lo / scale), 0, 15)
 *     q     = clamp(round(w / scale) + zero, 0, 15)
 *     w_hat = (q - zero) * scale
 *   and the product y[m][n] = sum_k w_hat[n][k] * x[m][k], evaluated per group
 *   as scale * (sum q*x - zero * sum x) without materialising w_hat in HBM.
 *   "round" rounds halfway cases away from zero; every division is an IEEE f32
 *   division.
 *
 * Shapes and layouts (all row-major):
 *   W       f32 [N][K]           K % 128 == 0, N >= 1
 *   packed  u8  [N][K/2]         canonical layout: two codes per byte, the
 *                                even k in the low nibble (page, "Code")
 *   scale   f32 [N][K/128]       canonical
 *   zero    u8  [N][K/128]       canonical
 *   qw      opaque device buffer of q4_weight_bytes(N, K, layout) bytes
 *           holding the same codes, scales and zeros in one of the kernels'
 *           tiled layouts: Q4_LAYOUT_TILED (f32 scales, u8 zeros; written by
 *           q4_repack, read back by q4_unpack) or Q4_LAYOUT_COMPACT (binary16
 *           scales, 4-bit zeros; q4_repack_compact)
 *   x       [M][K] of dtype xt,  y  [M][N] of dtype yt
 *
 * A second quantizer, q4_quantize_sym, follows the symmetric scheme of the
 * page "Quantization" (max|w| / 7 scales, codes stored with zero 8), into
 * the same canonical arrays.
 *
 * Conventions shared by every entry point:
 *   - All pointers are device pointers unless stated; the caller owns all
 *     memory.  No entry point allocates, frees or synchronises (except
 *     q4_check), and every one is asynchronous on `stream` (NULL = the legacy
 *     default stream).
 *   - Argument errors are detected on the host before anything is launched,
 *     and nothing is written: Q4_ERR_INVALID_ARG (bad sizes, NULL pointers,
 *     K % 128 != 0, a weight buffer whose size does not match its layout,
 *     short workspace), Q4_ERR_UNSUPPORTED (M or dtype outside
 *     what the entry point handles), Q4_ERR_MISALIGNED (a pointer without the
 *     alignment stated for it).
 *   - A failed launch returns Q4_ERR_CUDA (the CUDA error text is kept for
 *     q4_last_cuda_error).  There is no fallback path of any kind.
 *   - Weights must be finite; NaN or infinite weights give unspecified codes.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *q4_stream_t; /* same type as cudaStream_t */

typedef enum {
    Q4_OK = 0,
    Q4_ERR_INVALID_ARG = 1,
    Q4_ERR_UNSUPPORTED = 2,
    Q4_ERR_MISALIGNED = 3,
    Q4_ERR_CUDA = 4,
    Q4_ERR_TIMEOUT = 5,
    Q4_ERR_BOUNDS = 6
} q4_status;

typedef enum { Q4_F32 = 0, Q4_BF16 = 1, Q4_F16 = 2 } q4_dtype;

/* How a weight buffer `qw` holds its codes, scales and zeros (the two tiled
 * layouts written by q4_repack and q4_repack_compact below).  The products
 * take the layout and the buffer's byte count with every call and reject a
 * buffer whose size does not match that layout for (N, K): a compact buffer
 * handed over as TILED, or one written for another shape, is refused before
 * any launch instead of being read past its end (page "Weight quantization",
 * section "Pitfalls": converting without repacking gives garbage that still
 * runs; page "LLM Quantization Architecture in Depth", section "Kernels and
 * memory layout": the format is a contract). */
typedef enum { Q4_LAYOUT_TILED = 1, Q4_LAYOUT_COMPACT = 2 } q4_layout;

#define Q4_GROUP 128
#define Q4_TILE_ROWS 16
#define Q4_TILE_BYTES 1104 /* 16 rows x 128 k: 1024 B codes + 64 B scales + 16 B zeros */
#define Q4_CMP_TILE_BYTES 1072 /* compact: 1024 B codes + 32 B binary16 scales + 8 B zeros + 8 B pad */
#define Q4_GEMV_MAX_M 16

/*
 * Round-to-nearest quantization and nibble packing of a row-major f32 matrix
 * (page "Weight quantization": "How it works" formulas, function `quantize`).
 * w: [N][K] f32, 16-byte aligned.  Writes packed [N][K/2], scale [N][K/128],
 * zero [N][K/128] (canonical layout).  Bit-identical to the page's f32
 * arithmetic: IEEE division, ties away from zero, no contraction.
 * Errors: INVALID_ARG for N < 1, K < 128, K % 128 != 0 or a NULL pointer;
 * MISALIGNED unless w is 16-byte aligned.
 */
q4_status q4_quantize(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                      uint8_t *zero, q4_stream_t stream);

/*
 * Symmetric variant (page "Quantization", hritesh-sonawane.github.io notes,
 * sections "How it really works" and "Code", int_quant; page "LLM
 * Quantization Architecture in Depth", the group-wise symmetric listing):
 * per group of 128, scale = max|w| / 7 in IEEE f32 (1 when that quotient is
 * 0) and q = clamp(round(w / scale), -8, 7) with ties to even.  Writes the
 * same canonical arrays as q4_quantize: code q + 8 in each nibble and zero 8,
 * so (code - zero) * scale = q * scale and q4_repack, q4_gemv and q4_gemm
 * serve it unchanged.  Same arguments and errors as q4_quantize.
 */
q4_status q4_quantize_sym(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                          uint8_t *zero, q4_stream_t stream);

/* Bytes of a weight buffer for an N x K matrix in `layout`: ceil(N/16) row
 * tiles times K/128 groups times Q4_TILE_BYTES (TILED) or Q4_CMP_TILE_BYTES
 * (COMPACT).  0 for invalid sizes or an unknown layout. */
size_t q4_weight_bytes(int64_t N, int64_t K, q4_layout layout);

/*
 * Canonical -> tiled kernel layout ("packed formats with scale interleaving",
 * page "quant_llm_arch_2k", section "Memory Layout"; the offline pre-shuffle
 * of page "Weight quantization", section "Code", closing remark).  A
 * bijection: q4_unpack inverts it exactly.  Rows N..16*ceil(N/16)-1 of the
 * last tile are written as zeros.  qw must be 16-byte aligned and hold
 * q4_weight_bytes(N, K, Q4_LAYOUT_TILED) bytes; it may not overlap the
 * inputs.
 * Tile order (both tiled layouts): blocks of 8 row tiles (128 rows); inside
 * a block, steps of 4 groups (512 k); inside a step, row tile then group.
 * With T = ceil(N/16) row tiles and NG = K/128 groups, tile (row tile rt,
 * group g) is tile number
 *     8*NG*b + nb*4*s + (rt - 8b)*ns + (g - 4s)
 * where b = rt/8, s = g/4, nb = min(8, T - 8b) (row tiles in block b) and
 * ns = min(4, NG - 4s) (groups in step s): one step of one block, which a
 * decode GEMV reads as a unit, is one contiguous run of tiles.  Row-wise
 * concatenation of two buffers is the buffer of the stacked matrix when the
 * first has a multiple of 128 rows.
 * Tile number t starts at byte t * 1104:
 *   bytes [0, 1024): 32 lanes x 2 chunks of 16 B; chunk c of lane l = 4 words,
 *     word i covers k-step j = 4c+i (k = 128g + 16j .. +15) for tile rows
 *     r = l/4 and r+8 and k offsets 2(l%4) + {0,1,8,9}; nibble fields (bit
 *     offset: row, k offset) 0:(r,0) 16:(r,1) 4:(r+8,0) 20:(r+8,1)
 *     8:(r+8,8) 24:(r+8,9) 12:(r,8) 28:(r,9)
 *   bytes [1024, 1088): f32 scale pairs (s[i], s[i+8]) for i = 0..7
 *   bytes [1088, 1104): u8 zero pairs (z[i], z[i+8]) for i = 0..7
 */
q4_status q4_repack(const uint8_t *packed, const float *scale, const uint8_t *zero, int64_t N,
                    int64_t K, void *qw, q4_stream_t stream);

/* Tiled kernel layout -> canonical layout (exact inverse of q4_repack). */
q4_status q4_unpack(const void *qw, int64_t N, int64_t K, uint8_t *packed, float *scale,
                    uint8_t *zero, q4_stream_t stream);

/*
 * Compact metadata (page "Weight quantization": its printed bits per weight
 * count 16-bit scales and 4-bit zeros, "Complexity and constants" names the
 * fp16 scale + 4-bit zero format, "Implementation notes" keep scales in
 * fp16/bf16).  Same codes and zeros as the canonical arrays; each scale is
 * stored as IEEE binary16 rounded to nearest even (scales must lie in
 * binary16's normal range, 6.1e-5 .. 65504, to keep their precision), so
 * w_hat = (q - zero) * fp16(scale).  Tiles in the order above, tile number
 * t at byte t * 1072: bytes [0, 1024) codes exactly as in the tiled layout above; [1024,
 * 1056) binary16 scale pairs (s[i], s[i+8]) for i = 0..7; [1056, 1064) one
 * byte per pair, z[i] | z[i+8] << 4; [1064, 1072) zero padding (every tile
 * stays 16-byte aligned).  4.1875 bits per weight in memory.
 *
 * The buffer holds q4_weight_bytes(N, K, Q4_LAYOUT_COMPACT) bytes, and the
 * products read it when called with Q4_LAYOUT_COMPACT.
 * q4_repack_compact: canonical -> compact tiles; arguments, alignment and
 *   errors as q4_repack.
 * q4_unpack_compact: compact tiles -> codes [N][K/2], binary16 scale bits
 *   scale16 [N][K/128], zeros [N][K/128] (one byte per group).
 */
q4_status q4_repack_compact(const uint8_t *packed, const float *scale, const uint8_t *zero,
                            int64_t N, int64_t K, void *qw, q4_stream_t stream);
q4_status q4_unpack_compact(const void *qw, int64_t N, int64_t K, uint8_t *packed,
                            uint16_t *scale16, uint8_t *zero, q4_stream_t stream);

/*
 * Activation group sums, xsum[m][g] = sum_{k in group g} x[m][k] accumulated
 * in f32 (the "sum x" of the factored group dot, page "Weight quantization",
 * "How it works").  x: [M][K] of dtype xt; xsum: f32 [M][K/128].
 */
q4_status q4_xsum(const void *x, q4_dtype xt, int64_t M, int64_t K, float *xsum,
                  q4_stream_t stream);

/* Workspace bytes q4_gemv needs for this problem on the current device (0
 * when no split over K is used), whatever the activation type, path or
 * layout.  Layout: split-K arrival counters (one u32 per 32 output rows,
 * padded to 256 B) followed by f32 partial sums.
 *
 * Workspace rule (q4_gemv, q4_gemm): zero-fill a workspace once after
 * allocating it.  Every call that completes leaves the bytes it used zero
 * again (the CTA that finishes a split row block clears the counter and the
 * partial sums it consumed), so one workspace of the largest size needed
 * may serve any sequence of calls on one stream -- any shape, type or
 * layout, GEMV and GEMM alike.  Calls that may run at the same time on the
 * GPU (other streams) need separate workspaces.  After a call whose bounded
 * wait ran out (q4_check returns Q4_ERR_TIMEOUT) zero it again. */
size_t q4_gemv_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Decode GEMV, 1 <= M <= 16:  y[m][n] = sum over groups g of
 *   scale[n][g] * (sum_{k in g} q[n][k] * x[m][k] - zero[n][g] * sum_{k in g} x[m][k])
 * (page "Weight quantization", "How it works", factored group dot; function
 * `dot`), fp32 accumulation, dequantization fused in registers.
 * x: [M][K] (xt = F32, BF16 or F16); qw: a weight buffer in `layout`
 * (q4_repack: Q4_LAYOUT_TILED; q4_repack_compact: Q4_LAYOUT_COMPACT) of
 * qw_bytes bytes, which must equal q4_weight_bytes(N, K, layout); y: [M][N]
 * (yt = F32, BF16 or F16, rounded to nearest even from f32).
 * x, qw, y and workspace must be 16-byte aligned; workspace may be NULL when
 * q4_gemv_workspace_bytes returns 0.  Errors: UNSUPPORTED for M outside
 * [1, 16]; INVALID_ARG for bad sizes, an unknown layout, a qw_bytes that
 * does not match the layout and shape, or a short workspace.
 * Weights are read as constants: the kernel starts copying qw before it
 * waits for the previous kernel on the stream to finish (programmatic
 * dependent launch).  That is safe after any stream work that does not
 * trigger dependent launches early -- copies, memsets, ordinary kernels,
 * and every kernel of this library that writes a weight buffer -- but qw
 * must not be written by a kernel that calls
 * cudaTriggerProgrammaticLaunchCompletion (griddepcontrol.launch_dependents)
 * before its writes are done.
 */
q4_status q4_gemv(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K, const void *qw,
                  q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt, void *workspace,
                  size_t workspace_bytes, q4_stream_t stream);

/* Kernel choice for q4_gemv_path.  FMA: CUDA-core f32 FMAs on codes turned
 * into f32 in registers (M = 1 only).  MMA: m16n8k16 tensor-core MMAs with the
 * codes as bf16/f16 A fragments built in registers and the batch as the n
 * dimension (f32 activations as a bf16 high part plus a bf16 low part, two
 * MMAs per fragment).  AUTO (what q4_gemv uses): MMA. */
#define Q4_PATH_AUTO 0
#define Q4_PATH_FMA 1
#define Q4_PATH_MMA 2

/* q4_gemv with an explicit kernel choice (same arguments, same results within
 * the f32 accumulation tolerance).  UNSUPPORTED for FMA with M != 1 or with
 * compact tiles. */
q4_status q4_gemv_path(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                       const void *qw, q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt,
                       void *workspace, size_t workspace_bytes, int path, q4_stream_t stream);

/* Diagnostic for the bounded-wait machinery: launches the q4_gemv kernel for
 * this problem with its copy engine told to issue nothing, so every consumer
 * wait runs out after 20 ms.  The kernel then writes no output and raises the
 * device error word; a following q4_check(stream) returns Q4_ERR_TIMEOUT.
 * No GPU fault is involved and the context stays usable. */
q4_status q4_gemv_timeout_selftest(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                                   const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                                   q4_dtype yt, void *workspace, size_t workspace_bytes,
                                   q4_stream_t stream);

/*
 * Large-M W4A16 GEMM, Y[M][N] = X[M][K] * W_hat[N][K]^T (prefill; page
 * "LLM Quantization Architecture in Depth", section "Kernels and memory
 * layout": the kernel loads packed codes and scales, dequantizes on chip and
 * feeds the tensor cores in the same pass).  Both tensor-core operands are
 * binary16 behind exact powers of two: each weight row is scaled by 2^-e[n]
 * (15 * its largest group scale lands in [2^14, 2^15)) and each weight
 * w_hat = scale * (q - zero) is rounded once to binary16 (relative error at
 * most 2^-11); each token row is scaled by 2^-a[m] (its largest |x| lands
 * in the same range) and converted exactly.  The tcgen05 tensor cores
 * accumulate in f32 and the result is scaled back by 2^(e[n] + a[m]).  So
 * |Y - exact| <= 2^-11 * sum |w_hat x| + f32 accumulation, within the page's
 * 1e-3 * sum |w_hat x| at any K.  (A group whose scale is more than 2^20
 * below its row's largest, or a token row whose |x| spans more than about
 * 2^31, loses the excess precision to binary16's subnormal range.)
 * One call runs three passes on `stream`: the normalizations and, for bf16
 * activations, the binary16 copy of x into the workspace; the GEMM kernel;
 * the scratch part of the workspace set back to zero.
 * x: [M][K] BF16 or F16 (16-byte aligned); qw: as for q4_gemv; y: [M][N]
 * BF16, F16 or F32.  Any M >= 1 and N >= 1.  Each CTA tile covers 128
 * weight rows and the smallest of 16, 32, 64 or 128 tokens that covers M
 * (128 beyond, or 256 when 256-token tiles alone give every SM eight or
 * more); when the tiles are too few to fill the GPU, the groups of a
 * tile are split over several CTAs and their f32 partial sums added in a
 * fixed order through the workspace.  Workspace: q4_gemm_workspace_bytes
 * (always needed; the workspace rule of q4_gemv_workspace_bytes applies).
 * Errors as q4_gemv (UNSUPPORTED for F32 activations).
 */
q4_status q4_gemm(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K, const void *qw,
                  q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt, void *workspace,
                  size_t workspace_bytes, q4_stream_t stream);

/* Workspace bytes q4_gemm needs for this problem on the current device:
 * one u32 arrival counter per tile, padded to 256 B, and f32 partial sums
 * (only when tiles are split over CTAs), then the scratch of the first pass
 * (row and token factors, f32; the binary16 copy of x, 2 * M * K bytes),
 * each part 1024-byte aligned.  Same rule as q4_gemv_workspace_bytes: a
 * completed call leaves all of it zero. */
size_t q4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Diagnostic for the GEMM's bounded waits: launches q4_gemm's kernel with
 * its weight copies switched off, so the dequantizing warps' waits run out
 * after 20 ms; every role then stops, the CTA waits for the copies and
 * tensor-core operations it has in flight, frees its tensor memory and
 * returns without writing y.  A following q4_check(stream) returns
 * Q4_ERR_TIMEOUT; no GPU fault is involved and the context stays usable. */
q4_status q4_gemm_timeout_selftest(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                                   const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                                   q4_dtype yt, void *workspace, size_t workspace_bytes,
                                   q4_stream_t stream);

/* Size of the static scratch array used by q4_gemv_noalloc (16 MiB; held on
 * every GPU that loads this library until the process exits). */
#define Q4_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * q4_gemv without a workspace argument, for callers that cannot allocate
 * device memory (a plugin whose host framework owns all device memory and
 * passes only inputs and outputs; a decode loop that must never call an
 * allocator; a process whose GPU memory is reserved by another allocator).
 * No counterpart on the pages: it exists only for those callers.
 * Same arguments and results as q4_gemv (same kernels), without the
 * workspace.  The workspace comes from a static device array of
 * Q4_NOALLOC_SCRATCH_BYTES; problems that need more return
 * Q4_ERR_UNSUPPORTED before any launch.  Allocates nothing.  The first call
 * on each device looks up the array's address with that device current
 * (make it before any stream capture).  All calls on a device share the
 * array and each clears the counter block it uses with an asynchronous
 * memset on `stream` (so a call after one that timed out starts clean);
 * calls that overlap on the GPU race, so order them.
 */
q4_status q4_gemv_noalloc(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                          const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                          q4_dtype yt, q4_stream_t stream);

/* Synchronises `stream` and reports errors raised on the device since the
 * last check: Q4_ERR_BOUNDS when, in a library built with -DQ4_DEBUG, a
 * kernel computed a global store outside the buffer it writes (the store was
 * skipped; release builds do not check), Q4_ERR_TIMEOUT when a bounded wait
 * inside a kernel gave up (the kernel then returned without writing its
 * outputs), Q4_ERR_CUDA for a CUDA error, else Q4_OK.  Clears the device
 * error word. */
q4_status q4_check(q4_stream_t stream);

/* Static description of a status code. */
const char *q4_status_str(q4_status status);

/* Self-test of the store checks of a -DQ4_DEBUG build.  `buf`: at least 32
 * bytes of device memory.  One kernel writes byte i = i + 1 for i in 0..31
 * through the same check the other kernels use, declaring an extent of 16
 * bytes: bytes 0..15 are written, bytes 16..31 are left as they were and the
 * device error word records the skipped stores (the next q4_check returns
 * Q4_ERR_BOUNDS).  Every store the kernel attempts lies inside the 32 bytes,
 * so the test is safe even if the check were wrong.  A release build returns
 * Q4_ERR_UNSUPPORTED and launches nothing. */
q4_status q4_debug_bounds_selftest(uint8_t *buf, q4_stream_t stream);

/* Text of the most recent CUDA error seen by this library in this thread. */
const char *q4_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* Q4_H */
