// q3_K decode GEMV: the one-lane-per-block kernel of gemv_q4K.cuh where the
// problem's geometry allows it (q4lane::lane_eligible), else the
// four-lanes-per-block kernel of gemv_impl.cuh.
#include "gemv_q4K.cuh"

namespace plm {

cudaError_t run_group_q3K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream) {
    return q4lane::run_group_words<3>(p, count, m, subdots, stream);
}

bool gemv_supported_q3K(int k) { return gemv_rows_per_pass<3>(1, k / QK) > 0; }

}  // namespace plm
