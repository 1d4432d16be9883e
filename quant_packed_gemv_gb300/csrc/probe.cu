// Diagnostic: measured issue rates of the warp-level tensor instructions
// that an int8 and an f16 contraction could use on this device (context for
// the tensor-core kernels: on GB300, sm_103a, tcgen05 has no int8 kind, and
// these legacy warp-level rates are far below the tcgen05 f16 dense rate the
// GEMM's roofline uses).  Register-only loops; the one store per thread goes
// to a static device word (nothing is allocated).  Also the failure-detection
// self-test of the bounded waits.
#include <cstdint>

#include "../../include/plm.h"
#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

static __device__ int g_probe_sink;

template <int KIND>
__global__ void __launch_bounds__(256) mma_rate_kernel(int iters) {
    uint32_t a0 = threadIdx.x, a1 = a0 * 3u, a2 = a0 * 5u, a3 = a0 * 7u, b0 = a0 ^ 0x55u, b1 = a0 ^ 0x33u;
    int acc[8][4] = {};
    float facc[8][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (KIND == 0)
                asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                             "{%8,%9}, {%0,%1,%2,%3};"
                             : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
                             : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
            else
                asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                             "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                             : "+f"(facc[c][0]), "+f"(facc[c][1]), "+f"(facc[c][2]), "+f"(facc[c][3])
                             : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
    }
    int s = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) s += acc[c][j] + (int)facc[c][j];
    if (s == 0x12345678) g_probe_sink = s;
}

template <int KIND>
static cudaError_t time_rate(double* out) {
    const int blocks = num_sms() * 4, threads = 256, iters = 4096;
    cudaEvent_t e0, e1;
    cudaError_t e = cudaEventCreate(&e0);
    if (e != cudaSuccess) return e;
    e = cudaEventCreate(&e1);
    if (e != cudaSuccess) { cudaEventDestroy(e0); return e; }
    float best = 1e30f;
    for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
        cudaEventRecord(e0, 0);
        mma_rate_kernel<KIND><<<blocks, threads, 0, 0>>>(iters);
        cudaEventRecord(e1, 0);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        float ms = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
        if (e == cudaSuccess && ms < best) best = ms;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    // ops per warp per mma: 2*M*N*K
    const double per_mma = KIND == 0 ? 2.0 * 16 * 8 * 32 : 2.0 * 16 * 8 * 16;
    const double ops = (double)blocks * (threads / 32) * iters * 8 * per_mma;
    *out = ops / (best * 1e-3) / 1e12;
    return cudaSuccess;
}

// Failure-detection self-test: one warp waits on an mbarrier of its own with
// the same bounded wait the streaming kernels use, limited to `rounds`
// rounds.  With complete != 0 the barrier's one arrival is made first, so the
// wait ends at once; otherwise nothing ever arrives (no copy is issued), the
// wait runs out and bit 0 of the fault word is set, exactly as a streaming
// kernel records a copy that never landed.  The kernel then returns.
__global__ void bounded_wait_kernel(unsigned rounds, int complete, unsigned* fault) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        if (complete) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(&bar)) : "memory");
        if (!mbar_wait(&bar, 0, rounds)) atomicOr(fault, 1u);
    }
}

}  // namespace plm

extern "C" plm_status plm_selftest_bounded_wait(uint32_t rounds, int complete, cudaStream_t stream) {
    if (rounds < 1 || rounds > plm::WAIT_LIMIT) return PLM_ERR_INVALID_ARG;
    unsigned* fault = plm::fault_word();
    if (!fault) return PLM_ERR_CUDA;
    plm::bounded_wait_kernel<<<1, 32, 0, stream>>>(rounds, complete ? 1 : 0, fault);
    return cudaGetLastError() == cudaSuccess ? PLM_OK : PLM_ERR_CUDA;
}

extern "C" plm_status plm_probe_mma_rates(double* s8_tops, double* f16_tflops) {
    if (!s8_tops || !f16_tflops) return PLM_ERR_INVALID_ARG;
    cudaError_t e = plm::time_rate<0>(s8_tops);
    if (e == cudaSuccess) e = plm::time_rate<1>(f16_tflops);
    if (e != cudaSuccess) return PLM_ERR_CUDA;
    return PLM_OK;
}
