// Prefill GEMM entry.  First version: the activation rows are taken eight at
// a time through the decode GEMV kernels (correct for any m; W is re-read
// once per group of eight rows).
#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

cudaError_t launch_gemm(int fmt, const uint8_t* w, const uint8_t* xq, float* y,
                        long long m, int n, int k, cudaStream_t stream) {
    const int nb = k / QK;
    for (long long i0 = 0; i0 < m; i0 += GEMV_MAX_M) {
        const int mm = (int)(m - i0 < GEMV_MAX_M ? m - i0 : GEMV_MAX_M);
        cudaError_t e = launch_gemv(fmt, w, xq + (size_t)i0 * nb * Q8K_BYTES, y + (size_t)i0 * n,
                                    mm, n, k, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace plm
