// q4_K decode GEMV on f32 activations, quantized to q8_K inside the kernel
// (the fused q8_K producer; kernel in gemv_q4K.cuh).
#include "gemv_q4K.cuh"

namespace plm {

cudaError_t run_group_q4K_f32(const HostProblem* probs, int count, int m, cudaStream_t stream) {
    return q4lane::run_group<4, true, false>(probs, count, m, false, stream);
}

}  // namespace plm
