// q4_K gate/up pair with the SwiGLU epilogue (kernel in gemv_q4K.cuh):
// h = silu(W_gate . x) * (W_up . x), both matrices streamed in one launch.
#include "gemv_q4K.cuh"

namespace plm {

cudaError_t run_group_q4K_swiglu(const HostProblem* probs, int count, int m, cudaStream_t stream) {
    return q4lane::run_group<4, false, true>(probs, count, m, false, stream);
}

}  // namespace plm
