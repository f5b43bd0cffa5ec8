// noalloc.cu -- q4_gemv_noalloc: the decode GEMV for callers that cannot
// allocate device memory.
//
// q4_gemv needs a caller-provided workspace when a row block's K range is
// shared by several CTAs (arrival counters + partial sums).  Some callers
// cannot provide one: a plugin or operator running inside a host framework
// that owns all device memory and hands over only its input and output
// buffers, a latency-critical decode loop that must never call into an
// allocator (cudaMalloc can block on device-wide synchronisation and can fail
// once a caching allocator has reserved the GPU), or a process whose device
// memory is fully reserved by another allocator.  This entry point uses a
// fixed scratch array in the library's own static device memory instead.
//
// Costs and rules of that choice:
//   * every GPU that loads this library holds Q4_NOALLOC_SCRATCH_BYTES of it
//     until the process exits;
//   * problems whose workspace would exceed that size are rejected with
//     Q4_ERR_UNSUPPORTED before anything is launched;
//   * all calls on a device share the one array, which keeps the last call's
//     contents: each call clears the counter block it relies on (an
//     asynchronous memset on the same stream, no allocation; completed calls
//     leave it zero anyway, this also covers one that timed out), and calls
//     that overlap on the GPU (e.g. concurrent streams) race on the array, so
//     callers must order them;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before starting any stream capture.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_q4_scratch[Q4_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (looked up once
// per device); nullptr with *err set on failure.
void *scratch_for_current_device(cudaError_t *err)
{
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_q4_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" q4_status q4_gemv_noalloc(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                                     const void *qw, q4_layout layout, size_t qw_bytes, void *y,
                                     q4_dtype yt, q4_stream_t stream)
{
    if (!x || !qw || !y) return Q4_ERR_INVALID_ARG;
    if (N < 1 || K < Q4_GROUP || K % Q4_GROUP != 0) return Q4_ERR_INVALID_ARG;
    if (M < 1 || M > Q4_GEMV_MAX_M) return Q4_ERR_UNSUPPORTED;
    // the weight buffer matches its layout and shape (checked again by q4_gemv)
    const size_t wb = q4_weight_bytes(N, K, layout);
    if (wb == 0 || qw_bytes != wb) return Q4_ERR_INVALID_ARG;
    const size_t need = q4_gemv_workspace_bytes(M, N, K);
    if (need > Q4_NOALLOC_SCRATCH_BYTES) return Q4_ERR_UNSUPPORTED;  // beyond the static maximum
    cudaError_t err = cudaSuccess;
    void *scratch = scratch_for_current_device(&err);
    if (!scratch) return q4::cuda_fail(err);
    if (need > 0) {
        // The arrival counters (one u32 per 32 output rows, padded to 256
        // bytes, at the start of the workspace) must start at zero.  A
        // completed call leaves them zero; this also covers a call that
        // ended in a bounded-wait timeout.
        const size_t counters = q4::gemv_counter_bytes(N);
        err = cudaMemsetAsync(scratch, 0, counters < need ? counters : need,
                              reinterpret_cast<cudaStream_t>(stream));
        if (err != cudaSuccess) return q4::cuda_fail(err);
    }
    return q4_gemv(x, xt, M, N, K, qw, layout, qw_bytes, y, yt, need > 0 ? scratch : nullptr, need,
                   stream);
}
