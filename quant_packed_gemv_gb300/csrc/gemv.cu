// Host dispatch of the decode GEMV: single problems, groups of problems and
// the sub-dot export, by block format.
#include "gemv_impl.cuh"

namespace plm {

cudaError_t run_group_q4K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream);
cudaError_t run_group_q4K_f32(const HostProblem* p, int count, int m, cudaStream_t stream);
cudaError_t run_group_q4K_swiglu(const HostProblem* p, int count, int m, cudaStream_t stream);
cudaError_t run_group_q2K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream);
cudaError_t run_group_q3K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream);
cudaError_t run_group_q5K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream);
cudaError_t run_group_q6K(const HostProblem* p, int count, int m, bool subdots, cudaStream_t stream);
bool gemv_supported_q2K(int k);
bool gemv_supported_q3K(int k);
bool gemv_supported_q4K(int k);
bool gemv_supported_q5K(int k);
bool gemv_supported_q6K(int k);

bool gemv_supported(int fmt, int k) {
    switch (fmt) {
        case 2: return gemv_supported_q2K(k);
        case 3: return gemv_supported_q3K(k);
        case 4: return gemv_supported_q4K(k);
        case 5: return gemv_supported_q5K(k);
        case 6: return gemv_supported_q6K(k);
        default: return false;
    }
}

static cudaError_t run_fmt(int fmt, const HostProblem* p, int count, int m, bool subdots, cudaStream_t s) {
    switch (fmt) {
        case 2: return run_group_q2K(p, count, m, subdots, s);
        case 3: return run_group_q3K(p, count, m, subdots, s);
        case 4: return run_group_q4K(p, count, m, subdots, s);
        case 5: return run_group_q5K(p, count, m, subdots, s);
        case 6: return run_group_q6K(p, count, m, subdots, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(int fmt, const uint8_t* w, const uint8_t* xq, float* y,
                        int m, int n, int k, cudaStream_t stream) {
    HostProblem p{w, xq, y, nullptr, n, k / QK};
    return run_fmt(fmt, &p, 1, m, false, stream);
}

cudaError_t launch_subdots(int fmt, const uint8_t* w, const uint8_t* xq, int32_t* out,
                           int m, int n, int k, cudaStream_t stream) {
    HostProblem p{w, xq, nullptr, out, n, k / QK};
    return run_fmt(fmt, &p, 1, m, true, stream);
}

cudaError_t launch_gemv_grouped(int fmt, const GroupItem* items, int count, int m, cudaStream_t stream) {
    HostProblem part[GROUP_MAX];
    for (int p0 = 0; p0 < count; p0 += GROUP_MAX) {
        const int cnt = count - p0 < GROUP_MAX ? count - p0 : GROUP_MAX;
        for (int j = 0; j < cnt; ++j) {
            const GroupItem& g = items[p0 + j];
            part[j] = HostProblem{g.w, g.xq, g.y, nullptr, g.n, g.k / QK};
        }
        const cudaError_t e = run_fmt(fmt, part, cnt, m, false, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv_q4K_swiglu(const GroupItem* items, int count, int m, cudaStream_t stream) {
    HostProblem part[GROUP_MAX];
    for (int p0 = 0; p0 < count; p0 += GROUP_MAX) {
        const int cnt = count - p0 < GROUP_MAX ? count - p0 : GROUP_MAX;
        for (int j = 0; j < cnt; ++j) {
            const GroupItem& g = items[p0 + j];
            part[j] = HostProblem{g.w, g.xq, g.y, nullptr, g.n, g.k / QK, g.w2};
        }
        const cudaError_t e = run_group_q4K_swiglu(part, cnt, m, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_quantize_gemv_q4K(const GroupItem* items, int count, int m, cudaStream_t stream) {
    HostProblem part[GROUP_MAX];
    for (int p0 = 0; p0 < count; p0 += GROUP_MAX) {
        const int cnt = count - p0 < GROUP_MAX ? count - p0 : GROUP_MAX;
        for (int j = 0; j < cnt; ++j) {
            const GroupItem& g = items[p0 + j];
            part[j] = HostProblem{g.w, g.xq, g.y, nullptr, g.n, g.k / QK};
        }
        const cudaError_t e = run_group_q4K_f32(part, cnt, m, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace plm
