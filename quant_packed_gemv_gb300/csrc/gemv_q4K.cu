// q4_K decode GEMV on q8_K activations (kernel in gemv_q4K.cuh).
#include "gemv_q4K.cuh"

namespace plm {

cudaError_t run_group_q4K(const HostProblem* probs, int count, int m, bool subdots, cudaStream_t stream) {
    return q4lane::run_group<4, false, false>(probs, count, m, subdots, stream);
}

// One activation row of the widest row must fit beside the smallest ring.
bool gemv_supported_q4K(int k) {
    return q4lane::align128((size_t)q4lane::seg_bytes<4>(k / QK)) + q4lane::ring_bytes<4>(12, 2) <=
           (size_t)smem_optin_bytes();
}

}  // namespace plm
