// q6_K decode GEMV.  The one-lane-per-block kernel of gemv_q4K.cuh takes a
// problem when its rows hold a multiple of eight blocks (k a multiple of
// 2048, so every stage copy starts and ends on a 16-byte boundary), its
// matrix starts on a 16-byte boundary and one activation row fits beside
// the kernel's smallest ring; the four-lanes-per-block kernel of
// gemv_impl.cuh takes the others.  The choice depends on the problem alone
// (not on m or on the other problems of a group), so a row's bits are the
// same for every m and every grouping.
#include "gemv_q4K.cuh"

namespace plm {

static bool lane_path(const HostProblem& p) {
    return p.nb % 8 == 0 && ((uintptr_t)p.w & 15u) == 0 &&
           q4lane::align128((size_t)q4lane::seg_bytes<6>(p.nb)) + q4lane::ring_bytes<6>(12, 2) <=
               (size_t)smem_optin_bytes();
}

cudaError_t run_group_q6K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream) {
    HostProblem lane[GROUP_MAX], quad[GROUP_MAX];
    int nl = 0, nq = 0;
    for (int i = 0; i < count; ++i) {
        if (lane_path(p[i]))
            lane[nl++] = p[i];
        else
            quad[nq++] = p[i];
    }
    cudaError_t e = cudaSuccess;
    if (nl > 0) e = q4lane::run_group<6, false, false>(lane, nl, m, subdots, stream);
    if (e == cudaSuccess && nq > 0) e = run_group<6>(quad, nq, m, subdots, stream);
    return e;
}

bool gemv_supported_q6K(int k) { return gemv_rows_per_pass<6>(1, k / QK) > 0; }

}  // namespace plm
