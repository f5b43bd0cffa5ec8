// api.cu -- the exported C ABI (include/q4.h): host-side argument checks,
// plan selection and launches.  Nothing here allocates or synchronises except
// q4_check.  Every product call names its weight layout and the weight
// buffer's byte count, checked against each other before anything runs.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

__device__ unsigned int g_q4_error = 0u;

namespace q4 {

static thread_local char t_last_error[256] = "";

q4_status cuda_fail(cudaError_t e)
{
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return Q4_ERR_CUDA;
}

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static inline bool valid_dtype(q4_dtype t) { return t == Q4_F32 || t == Q4_BF16 || t == Q4_F16; }

// Per-device cached facts.
struct DevInfo {
    int sm_count = 0;
    unsigned int *err = nullptr;
};
static std::mutex g_mu;
static DevInfo g_dev[64];

static const DevInfo *dev_info()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    DevInfo &d = g_dev[dev];
    if (d.sm_count == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_q4_error) != cudaSuccess) return nullptr;
        d.err = static_cast<unsigned int *>(p);
        d.sm_count = sms;
    }
    return &d;
}

unsigned int *device_error_word()
{
    const DevInfo *d = dev_info();
    return d ? d->err : nullptr;
}

// The error word for the store checks of the packing kernels: looked up
// only in debug builds, so release calls stay free of the device query.
static inline unsigned int *debug_err() { return kDebugBounds ? device_error_word() : nullptr; }

// Stores i + 1 into byte i of a 32-byte buffer through the store check,
// declaring an extent of 16.
__global__ void k_bounds_selftest(uint8_t *buf, unsigned int *err)
{
    const int i = threadIdx.x;
    if (i < 32 && store_ok(i, 16, err)) buf[i] = static_cast<uint8_t>(i + 1);
}

static inline bool sizes_ok(int64_t N, int64_t K)
{
    return N >= 1 && K >= G && K % G == 0 && N <= (1LL << 30) && K <= (1LL << 30) &&
           N * K <= (1LL << 40);
}

size_t weight_bytes(int64_t N, int64_t K, q4_layout layout)
{
    if (!sizes_ok(N, K)) return 0;
    const size_t tile = layout == Q4_LAYOUT_TILED ? TILE_BYTES
                        : layout == Q4_LAYOUT_COMPACT ? CMP_TILE_BYTES
                                                      : 0;
    return static_cast<size_t>((N + TILE_ROWS - 1) / TILE_ROWS) * static_cast<size_t>(K / G) * tile;
}

// The weight buffer matches its declared layout and shape byte for byte.
static inline bool weights_ok(int64_t N, int64_t K, q4_layout layout, size_t qw_bytes)
{
    const size_t need = weight_bytes(N, K, layout);
    return need != 0 && qw_bytes == need;
}

static q4_status gemv_common(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                             const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                             q4_dtype yt, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, int path, int debug_no_copy, uint64_t wait_ns)
{
    if (!x || !qw || !y) return Q4_ERR_INVALID_ARG;
    if (!sizes_ok(N, K) || N > (1LL << 28)) return Q4_ERR_INVALID_ARG;
    if (!weights_ok(N, K, layout, qw_bytes)) return Q4_ERR_INVALID_ARG;
    const bool cmp = layout == Q4_LAYOUT_COMPACT;
    if (M < 1 || M > Q4_GEMV_MAX_M) return Q4_ERR_UNSUPPORTED;
    if (!valid_dtype(xt) || !valid_dtype(yt)) return Q4_ERR_UNSUPPORTED;
    if (path == PATH_FMA && (M != 1 || cmp)) return Q4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(y) || !aligned16(workspace))
        return Q4_ERR_MISALIGNED;
    const DevInfo *d = dev_info();
    if (!d) return cuda_fail(cudaGetLastError());
    const GemvPlan plan = gemv_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                    xt, path, d->sm_count, cmp);
    if (plan.workspace > 0 && (!workspace || workspace_bytes < plan.workspace))
        return Q4_ERR_INVALID_ARG;
    GemvArgs a{};
    a.x = x;
    a.xt = xt;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.qw = static_cast<const uint8_t *>(qw);
    a.y = y;
    a.yt = yt;
    a.maxc = plan.maxc;
    if (plan.maxc > 1) {
        const size_t counters = gemv_counter_bytes(N);
        a.count = static_cast<unsigned int *>(workspace);
        a.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + counters);
        // store checks use the plan's own extents (inside the caller's buffer)
        a.count_len = plan.nrb;
        a.partial_len = static_cast<int64_t>((plan.workspace - counters) / sizeof(float));
    }
    a.wait_ns = wait_ns;
    a.err = d->err;
    a.debug_no_copy = debug_no_copy;
    const cudaError_t e = gemv_launch(plan, a, stream);
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

}  // namespace q4

using namespace q4;

extern "C" {

static q4_status quantize_common(const float *w, int64_t N, int64_t K, uint8_t *packed,
                                 float *scale, uint8_t *zero, bool symmetric, q4_stream_t stream)
{
    if (!w || !packed || !scale || !zero || !sizes_ok(N, K)) return Q4_ERR_INVALID_ARG;
    if (!aligned16(w)) return Q4_ERR_MISALIGNED;
    const cudaError_t e = quantize_launch(w, N, K, packed, scale, zero, symmetric, debug_err(),
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

q4_status q4_quantize(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                      uint8_t *zero, q4_stream_t stream)
{
    return quantize_common(w, N, K, packed, scale, zero, false, stream);
}

q4_status q4_quantize_sym(const float *w, int64_t N, int64_t K, uint8_t *packed, float *scale,
                          uint8_t *zero, q4_stream_t stream)
{
    return quantize_common(w, N, K, packed, scale, zero, true, stream);
}

size_t q4_weight_bytes(int64_t N, int64_t K, q4_layout layout)
{
    return weight_bytes(N, K, layout);
}

q4_status q4_repack(const uint8_t *packed, const float *scale, const uint8_t *zero, int64_t N,
                    int64_t K, void *qw, q4_stream_t stream)
{
    if (!packed || !scale || !zero || !qw || !sizes_ok(N, K)) return Q4_ERR_INVALID_ARG;
    if (!aligned16(qw)) return Q4_ERR_MISALIGNED;
    const cudaError_t e = repack_launch(packed, scale, zero, N, K, static_cast<uint8_t *>(qw),
                                        debug_err(), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

q4_status q4_unpack(const void *qw, int64_t N, int64_t K, uint8_t *packed, float *scale,
                    uint8_t *zero, q4_stream_t stream)
{
    if (!packed || !scale || !zero || !qw || !sizes_ok(N, K)) return Q4_ERR_INVALID_ARG;
    if (!aligned16(qw)) return Q4_ERR_MISALIGNED;
    const cudaError_t e = unpack_launch(static_cast<const uint8_t *>(qw), N, K, packed, scale,
                                        zero, debug_err(), reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

q4_status q4_repack_compact(const uint8_t *packed, const float *scale, const uint8_t *zero,
                            int64_t N, int64_t K, void *qw, q4_stream_t stream)
{
    if (!packed || !scale || !zero || !qw || !sizes_ok(N, K)) return Q4_ERR_INVALID_ARG;
    if (!aligned16(qw)) return Q4_ERR_MISALIGNED;
    const cudaError_t e = repack_compact_launch(packed, scale, zero, N, K,
                                                static_cast<uint8_t *>(qw), debug_err(),
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

q4_status q4_unpack_compact(const void *qw, int64_t N, int64_t K, uint8_t *packed,
                            uint16_t *scale16, uint8_t *zero, q4_stream_t stream)
{
    if (!packed || !scale16 || !zero || !qw || !sizes_ok(N, K)) return Q4_ERR_INVALID_ARG;
    if (!aligned16(qw)) return Q4_ERR_MISALIGNED;
    const cudaError_t e = unpack_compact_launch(static_cast<const uint8_t *>(qw), N, K, packed,
                                                scale16, zero, debug_err(),
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

q4_status q4_xsum(const void *x, q4_dtype xt, int64_t M, int64_t K, float *xsum,
                  q4_stream_t stream)
{
    if (!x || !xsum || M < 1 || !sizes_ok(M, K)) return Q4_ERR_INVALID_ARG;
    if (!valid_dtype(xt)) return Q4_ERR_UNSUPPORTED;
    const cudaError_t e = xsum_launch(x, xt, M, K, xsum, debug_err(),
                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

size_t q4_gemv_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || M > Q4_GEMV_MAX_M || !sizes_ok(N, K)) return 0;
    const DevInfo *d = dev_info();
    if (!d) return 0;
    // the largest need over activation types and paths, so one buffer serves
    // every call with this shape
    size_t need = 0;
    const q4_dtype types[3] = {Q4_BF16, Q4_F16, Q4_F32};
    const int paths[3] = {PATH_AUTO, PATH_MMA, PATH_FMA};
    for (int cmp = 0; cmp < 2; ++cmp)
        for (q4_dtype t : types)
            for (int p : paths) {
                if (p == PATH_FMA && (M != 1 || cmp)) continue;
                const GemvPlan g = gemv_plan(static_cast<int>(M), static_cast<int>(N),
                                             static_cast<int>(K), t, p, d->sm_count, cmp != 0);
                need = std::max(need, g.workspace);
            }
    return need;
}

q4_status q4_gemv(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K, const void *qw,
                  q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt, void *workspace,
                  size_t workspace_bytes, q4_stream_t stream)
{
    return gemv_common(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream), PATH_AUTO, 0, 1000000000ull);
}

q4_status q4_gemv_path(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                       const void *qw, q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt,
                       void *workspace, size_t workspace_bytes, int path, q4_stream_t stream)
{
    if (path != PATH_AUTO && path != PATH_FMA && path != PATH_MMA) return Q4_ERR_UNSUPPORTED;
    return gemv_common(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream), path, 0, 1000000000ull);
}

q4_status q4_gemv_timeout_selftest(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                                   const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                                   q4_dtype yt, void *workspace, size_t workspace_bytes,
                                   q4_stream_t stream)
{
    return gemv_common(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream), PATH_AUTO, 1, 20000000ull);
}

static q4_status gemm_common(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                             const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                             q4_dtype yt, void *workspace, size_t workspace_bytes,
                             q4_stream_t stream, int debug_no_copy, uint64_t wait_ns)
{
    if (!x || !qw || !y) return Q4_ERR_INVALID_ARG;
    if (M < 1 || M > (1LL << 30) || !sizes_ok(N, K) || N > (1LL << 30)) return Q4_ERR_INVALID_ARG;
    if (!weights_ok(N, K, layout, qw_bytes)) return Q4_ERR_INVALID_ARG;
    if ((xt != Q4_BF16 && xt != Q4_F16) || !valid_dtype(yt)) return Q4_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(qw) || !aligned16(y) || !aligned16(workspace))
        return Q4_ERR_MISALIGNED;
    const DevInfo *d = dev_info();
    if (!d) return cuda_fail(cudaGetLastError());
    const GemmPlan plan = gemm_plan(M, N, K, d->sm_count);
    if (plan.workspace > 0 && (!workspace || workspace_bytes < plan.workspace))
        return Q4_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    const q4_status st = gemm_run(plan, x, xt, M, N, K, static_cast<const uint8_t *>(qw),
                                  layout == Q4_LAYOUT_COMPACT, y, yt, workspace, d->err, wait_ns,
                                  debug_no_copy, reinterpret_cast<cudaStream_t>(stream), &e);
    if (st == Q4_ERR_CUDA) return cuda_fail(e);
    return st;
}

q4_status q4_gemm(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K, const void *qw,
                  q4_layout layout, size_t qw_bytes, void *y, q4_dtype yt, void *workspace,
                  size_t workspace_bytes, q4_stream_t stream)
{
    return gemm_common(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, workspace, workspace_bytes,
                       stream, 0, 2000000000ull);
}

size_t q4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || M > (1LL << 30) || !sizes_ok(N, K) || N > (1LL << 30)) return 0;
    const DevInfo *d = dev_info();
    if (!d) return 0;
    return gemm_plan(M, N, K, d->sm_count).workspace;
}

q4_status q4_gemm_timeout_selftest(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                                   const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                                   q4_dtype yt, void *workspace, size_t workspace_bytes,
                                   q4_stream_t stream)
{
    return gemm_common(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, workspace, workspace_bytes,
                       stream, 1, 20000000ull);
}

q4_status q4_check(q4_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_q4_error, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e);
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_q4_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
        return (word & ERR_BOUNDS) ? Q4_ERR_BOUNDS : Q4_ERR_TIMEOUT;
    }
    return Q4_OK;
}

const char *q4_status_str(q4_status status)
{
    switch (status) {
    case Q4_OK: return "ok";
    case Q4_ERR_INVALID_ARG: return "invalid argument";
    case Q4_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case Q4_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case Q4_ERR_CUDA: return "CUDA error";
    case Q4_ERR_TIMEOUT: return "a bounded device wait timed out";
    case Q4_ERR_BOUNDS: return "a store outside its buffer was skipped (debug build)";
    }
    return "unknown status";
}

const char *q4_last_cuda_error(void) { return t_last_error; }

q4_status q4_debug_bounds_selftest(uint8_t *buf, q4_stream_t stream)
{
    if (!kDebugBounds) return Q4_ERR_UNSUPPORTED;
    if (!buf) return Q4_ERR_INVALID_ARG;
    const DevInfo *d = dev_info();
    if (!d) return cuda_fail(cudaGetLastError());
    k_bounds_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(buf, d->err);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? Q4_OK : cuda_fail(e);
}

}  // extern "C"
