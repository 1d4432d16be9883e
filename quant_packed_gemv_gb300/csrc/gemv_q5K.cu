// q5_K decode GEMV (the one-lane-per-block kernel of gemv_q4K.cuh with the
// fifth bit of every weight taken from qh[32]).
#include "gemv_q4K.cuh"

namespace plm {

cudaError_t run_group_q5K(const HostProblem* probs, int count, int m, bool subdots, cudaStream_t stream) {
    return q4lane::run_group<5, false, false>(probs, count, m, subdots, stream);
}

// One activation row of the widest row must fit beside the smallest ring.
bool gemv_supported_q5K(int k) {
    return q4lane::align128((size_t)q4lane::seg_bytes<5>(k / QK)) + q4lane::ring_bytes<5>(12, 2) <=
           (size_t)smem_optin_bytes();
}

}  // namespace plm
