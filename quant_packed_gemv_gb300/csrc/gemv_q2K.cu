// q2K instantiation of the generic decode GEMV (kernel in gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace plm {

cudaError_t run_group_q2K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream) {
    return run_group<2>(p, count, m, subdots, stream);
}

bool gemv_supported_q2K(int k) { return gemv_rows_per_pass<2>(1, k / QK) > 0; }

}  // namespace plm
