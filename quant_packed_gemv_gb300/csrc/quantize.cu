// q8_K activation quantization (the int8 activation step of the packed
// matmul, PocketLLM "Current status" table, row "src/": one 256-element
// block per task).  One warp per 256-element chunk, 8 values per lane.
//
// The arithmetic is q8K_quantize_warp (plm_device.cuh), shared with the
// fused quantize + GEMV so that both give the same codes bit for bit.
#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

__global__ void __launch_bounds__(256) quantize_q8K_kernel(const float* __restrict__ x,
                                                           uint8_t* __restrict__ xq,
                                                           long long nchunks) {
    grid_launch_dependents();
    grid_wait_prior();
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long ch = warp0; ch < nchunks; ch += nwarps) {
        const float4* src = reinterpret_cast<const float4*>(x + ch * QK) + 2 * lane;
        const float4 a = __ldg(src), b = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};

        uint8_t* blk = xq + ch * Q8K_BYTES;
        int q[8];
        const float d = q8K_quantize_warp(v, lane, q);
        uint32_t w0, w1;
        pack_codes8(q, w0, w1);
        uint32_t* qsw = reinterpret_cast<uint32_t*>(blk + 4) + 2 * lane;
        qsw[0] = w0;
        qsw[1] = w1;
        // bsums: group g = lanes 2g, 2g+1
        int s = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
        const int s_next = __shfl_down_sync(0xFFFFFFFFu, s, 2);
        if ((lane & 3) == 0) {   // lane 4h writes bsums[2h] and bsums[2h+1]
            const uint32_t packed = ((uint32_t)s & 0xFFFFu) | ((uint32_t)s_next << 16);
            reinterpret_cast<uint32_t*>(blk + 260)[lane >> 2] = packed;
        }
        if (lane == 0) *reinterpret_cast<float*>(blk) = d;
    }
}

cudaError_t launch_quantize_q8K(const float* x, uint8_t* xq, long long m, long long k,
                                cudaStream_t stream) {
    const long long nchunks = m * (k / QK);
    const int threads = 256;
    long long blocks = (nchunks + 7) / 8;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    return launch_kernel(quantize_q8K_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, x, xq, nchunks);
}

}  // namespace plm
