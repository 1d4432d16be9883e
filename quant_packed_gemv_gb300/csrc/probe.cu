// Diagnostic: measured issue rates of the warp-level tensor instructions
// that an int8 and an f16 contraction could use on this device (context for
// the tensor-core kernels: on GB300, sm_103a, tcgen05 has no int8 kind, and
// these legacy warp-level rates are far below the tcgen05 f16 dense rate the
// GEMM's roofline uses).  Register-only loops; the one store per thread goes
// to a static device word (nothing is allocated).  The rate of the tcgen05
// MMA the GEMM issues, alone and with an mbarrier wait after each commit.
// Also the failure-detection self-test of the bounded waits.
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

// tcgen05 MMA rate: one thread of one CTA issues `nmma` MMAs of the GEMM's
// shape (kind::f16, M = 128, N = 128, K = 16, f32 accumulator in tensor
// memory, A from tensor memory, B from shared memory; zero operands) with a
// commit every four.  With WAIT, each commit is followed by an mbarrier wait
// on a phase that is already complete, as the GEMM's MMA thread waits for its
// next stage.  clock64 cycles from the first issue to the last commit's
// completion go to tc_cycles[blockIdx.x].  120 KB of shared memory keep one
// CTA per SM.
constexpr int TC_SMEM = 120 * 1024;
constexpr uint32_t TC_IDESC = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);   // f16 x f16 -> f32, 128 x 128
static __device__ unsigned long long tc_cycles[1024];

__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {   // K-major, 128-byte swizzle
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

template <bool WAIT>
__global__ void __launch_bounds__(128, 1) tc_rate_kernel(int nmma, unsigned* fault) {
    extern __shared__ __align__(1024) uint8_t tc_raw[];
    uint8_t* sm = tc_raw + ((1024u - (smem_u32(tc_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 16384);   // [0] last commit, [1] commits, [2] complete
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 4);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 16384 / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        mbar_arrive(&bars[2]);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(smem_u32(slot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the zero B tile, for the tensor core
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tm = *slot;
    {   // A: columns 256 .. 287 of every lane, zero
        const uint32_t z = 0u;
        asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
                     "%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                     :: "r"(tm + ((uint32_t)(warp * 32) << 16) + 256u), "r"(z) : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (threadIdx.x == 0) {
        const uint64_t db = tc_desc_sw128(smem_u32(sm));
        const unsigned long long t0 = clock64();
        bool ok = true;
        for (int i = 0; i < nmma && ok; ++i) {
            const int kk = i & 3;
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                         "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                         :: "r"(tm), "r"(tm + 256u + 8u * kk), "l"(db + 2 * kk), "r"(TC_IDESC), "r"((uint32_t)(i > 0)));
            if (kk == 3) {
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             :: "r"(smem_u32(&bars[1])) : "memory");
                if (WAIT) ok = mbar_wait(&bars[2], 0u);
            }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&bars[0])) : "memory");
        if (!mbar_wait(&bars[0], 0u)) ok = false;
        if (!ok) atomicOr(fault, 2u);
        tc_cycles[blockIdx.x] = clock64() - t0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tm) : "memory");
    }
}

template <bool WAIT>
static cudaError_t tc_rate(int grid, int nmma, double* cycles_per_mma, double* ms) {
    unsigned* fault = fault_word();
    if (!fault) return cudaErrorInvalidDevicePointer;
    cudaError_t e = cudaFuncSetAttribute(tc_rate_kernel<WAIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e != cudaSuccess) return e;
    cudaEvent_t e0, e1;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess) return e;
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) { cudaEventDestroy(e0); return e; }
    float best = 1e30f;
    for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {   // the first is a warm-up
        cudaEventRecord(e0, 0);
        tc_rate_kernel<WAIT><<<grid, 128, TC_SMEM, 0>>>(nmma, fault);
        cudaEventRecord(e1, 0);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventSynchronize(e1);
        float t = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
        if (e == cudaSuccess && rep > 0 && t < best) best = t;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return e;
    unsigned long long c[1024];
    if ((e = cudaMemcpyFromSymbol(c, tc_cycles, sizeof(unsigned long long) * grid)) != cudaSuccess) return e;
    double sum = 0.0;
    for (int i = 0; i < grid; ++i) sum += (double)c[i];
    *cycles_per_mma = sum / grid / nmma;
    *ms = best;
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

extern "C" plm_status plm_probe_tcgen05_rate(double* cycles_per_mma, double* cycles_per_mma_wait, double* tflops) {
    if (!cycles_per_mma || !cycles_per_mma_wait || !tflops) return PLM_ERR_INVALID_ARG;
    const int nmma = 4096, sms = plm::num_sms();
    if (sms < 1 || sms > 1024) return PLM_ERR_UNSUPPORTED;
    double ms = 0.0, unused = 0.0;
    cudaError_t e = plm::tc_rate<false>(1, nmma, cycles_per_mma, &ms);
    if (e == cudaSuccess) e = plm::tc_rate<true>(1, nmma, cycles_per_mma_wait, &ms);
    if (e == cudaSuccess) e = plm::tc_rate<false>(sms, nmma, &unused, &ms);
    if (e != cudaSuccess) return PLM_ERR_CUDA;
    *tflops = 2.0 * 128 * 128 * 16 * (double)nmma * sms / (ms * 1e-3) / 1e12;
    return PLM_OK;
}
