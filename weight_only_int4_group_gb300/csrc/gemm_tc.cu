// gemm_tc.cu -- large-M W4A16 GEMM on the tcgen05 tensor cores (in progress).
#include "common.cuh"

extern "C" q4_status q4_gemm(const void *x, q4_dtype xt, int64_t M, int64_t N, int64_t K,
                             const void *qw, void *y, q4_dtype yt, q4_stream_t stream)
{
    (void)x; (void)xt; (void)M; (void)N; (void)K; (void)qw; (void)y; (void)yt; (void)stream;
    return Q4_ERR_UNSUPPORTED;
}
