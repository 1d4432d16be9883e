// The C ABI of libplm: argument checks on the host, then one or more kernel
// launches on the caller's stream.  Nothing is allocated and nothing waits.
#include <atomic>
#include <cstdint>

#include "../../include/plm.h"
#include "plm_device.cuh"
#include "plm_internal.h"

namespace plm {

// Set (bitwise or) by kernels whose bounded wait on an asynchronous copy ran
// out; read and cleared by plm_device_fault.  One word per device, in the
// module's static device memory (nothing is allocated).
__device__ unsigned g_plm_fault = 0;

unsigned* fault_word() {
    // the symbol's address is fixed per device while the device's primary
    // context lives (the library must not be used across a cudaDeviceReset);
    // remember it for the first 64 devices.  Threads that race here store
    // the same address.
    static std::atomic<void*> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) {
        void* c = cache[dev].load(std::memory_order_acquire);
        if (c) return static_cast<unsigned*>(c);
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plm_fault) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < 64) cache[dev].store(p, std::memory_order_release);
    return static_cast<unsigned*>(p);
}

namespace {
std::atomic<int> g_overlap{1};
}
int overlap_mode() { return g_overlap.load(std::memory_order_relaxed); }

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    return n;
}

}  // namespace plm

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int64_t kMaxIndex = 0x7FFFFFFFLL;

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

plm_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PLM_OK;
    g_last_cuda_error = (int)e;
    return PLM_ERR_CUDA;
}

// Shape checks shared by the matmul entry points.
plm_status check_matmul(const void* w, const void* xq, const void* y, int64_t m, int64_t n,
                        int64_t k, int64_t max_m) {
    if (!w || !xq || !y) return PLM_ERR_INVALID_ARG;
    if (m <= 0 || n <= 0 || k <= 0 || k % plm::QK != 0) return PLM_ERR_INVALID_ARG;
    if (m > max_m || n > kMaxIndex || k > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (m * (k / plm::QK) > kMaxIndex || n * (k / plm::QK) > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(xq, 4) || !aligned(y, 4)) return PLM_ERR_MISALIGNED;
    return PLM_OK;
}

plm_status gemv_common(int fmt, const void* w, const void* xq, float* y, int64_t m, int64_t n,
                       int64_t k, cudaStream_t stream) {
    plm_status s = check_matmul(w, xq, y, m, n, k, plm::GEMV_MAX_M);
    if (s != PLM_OK) return s;
    if (!plm::gemv_supported(fmt, (int)k)) return PLM_ERR_UNSUPPORTED;
    return cuda_status(plm::launch_gemv(fmt, (const uint8_t*)w, (const uint8_t*)xq, y, (int)m,
                                        (int)n, (int)k, stream));
}

plm_status grouped_common(int fmt, const plm_gemv_problem* problems, int64_t count, int64_t m,
                          cudaStream_t stream) {
    if (!problems || count <= 0 || count > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (m <= 0 || m > plm::GEMV_MAX_M) return PLM_ERR_INVALID_ARG;
    constexpr int kChunk = 256;
    plm::GroupItem items[kChunk];
    // argument checks for every problem first, then size support
    for (int64_t j = 0; j < count; ++j) {
        const plm_gemv_problem& p = problems[j];
        plm_status s = check_matmul(p.w, p.xq, p.y, m, p.n, p.k, plm::GEMV_MAX_M);
        if (s != PLM_OK) return s;
    }
    for (int64_t j = 0; j < count; ++j)
        if (!plm::gemv_supported(fmt, (int)problems[j].k)) return PLM_ERR_UNSUPPORTED;
    for (int64_t p0 = 0; p0 < count; p0 += kChunk) {
        const int cnt = (int)(count - p0 < kChunk ? count - p0 : kChunk);
        for (int j = 0; j < cnt; ++j) {
            const plm_gemv_problem& p = problems[p0 + j];
            items[j] = plm::GroupItem{(const uint8_t*)p.w, (const uint8_t*)p.xq, p.y, (int)p.n, (int)p.k};
        }
        plm_status s = cuda_status(plm::launch_gemv_grouped(fmt, items, cnt, (int)m, stream));
        if (s != PLM_OK) return s;
    }
    return PLM_OK;
}

// Fused quantize + GEMV: f32 activations, 16-byte aligned for vector loads.
plm_status qgemv_common(const plm_qgemv_problem* problems, int64_t count, int64_t m, cudaStream_t stream) {
    if (!problems || count <= 0 || count > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (m <= 0 || m > plm::GEMV_MAX_M) return PLM_ERR_INVALID_ARG;
    for (int64_t j = 0; j < count; ++j) {
        const plm_qgemv_problem& p = problems[j];
        plm_status s = check_matmul(p.w, p.x, p.y, m, p.n, p.k, plm::GEMV_MAX_M);
        if (s != PLM_OK) return s;
        if (!aligned(p.x, 16)) return PLM_ERR_MISALIGNED;
    }
    for (int64_t j = 0; j < count; ++j)
        if (!plm::gemv_supported(4, (int)problems[j].k)) return PLM_ERR_UNSUPPORTED;
    constexpr int kChunk = 256;
    plm::GroupItem items[kChunk];
    for (int64_t p0 = 0; p0 < count; p0 += kChunk) {
        const int cnt = (int)(count - p0 < kChunk ? count - p0 : kChunk);
        for (int j = 0; j < cnt; ++j) {
            const plm_qgemv_problem& p = problems[p0 + j];
            items[j] = plm::GroupItem{(const uint8_t*)p.w, (const uint8_t*)p.x, p.y, (int)p.n, (int)p.k};
        }
        plm_status s = cuda_status(plm::launch_quantize_gemv_q4K(items, cnt, (int)m, stream));
        if (s != PLM_OK) return s;
    }
    return PLM_OK;
}

// Gate/up pairs: both matrices checked like a GEMV's weights.
plm_status swiglu_common(const plm_swiglu_problem* problems, int64_t count, int64_t m, cudaStream_t stream) {
    if (!problems || count <= 0 || count > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (m <= 0 || m > plm::GEMV_MAX_M) return PLM_ERR_INVALID_ARG;
    for (int64_t j = 0; j < count; ++j) {
        const plm_swiglu_problem& p = problems[j];
        plm_status s = check_matmul(p.w_gate, p.xq, p.h, m, p.n, p.k, plm::GEMV_MAX_M);
        if (s != PLM_OK) return s;
        s = check_matmul(p.w_up, p.xq, p.h, m, p.n, p.k, plm::GEMV_MAX_M);
        if (s != PLM_OK) return s;
    }
    for (int64_t j = 0; j < count; ++j)
        if (!plm::gemv_supported(4, (int)problems[j].k)) return PLM_ERR_UNSUPPORTED;
    constexpr int kChunk = 256;
    plm::GroupItem items[kChunk];
    for (int64_t p0 = 0; p0 < count; p0 += kChunk) {
        const int cnt = (int)(count - p0 < kChunk ? count - p0 : kChunk);
        for (int j = 0; j < cnt; ++j) {
            const plm_swiglu_problem& p = problems[p0 + j];
            items[j] = plm::GroupItem{(const uint8_t*)p.w_gate, (const uint8_t*)p.xq, p.h, (int)p.n, (int)p.k,
                                      (const uint8_t*)p.w_up};
        }
        plm_status s = cuda_status(plm::launch_gemv_q4K_swiglu(items, cnt, (int)m, stream));
        if (s != PLM_OK) return s;
    }
    return PLM_OK;
}

plm_status gemm_common(int fmt, const void* w, const void* xq, float* y, int64_t m, int64_t n,
                       int64_t k, cudaStream_t stream) {
    plm_status s = check_matmul(w, xq, y, m, n, k, kMaxIndex);
    if (s != PLM_OK) return s;
    if (m * n > (int64_t)1 << 40) return PLM_ERR_INVALID_ARG;
    if (!plm::gemv_supported(fmt, (int)k)) return PLM_ERR_UNSUPPORTED;
    return cuda_status(plm::launch_gemm(fmt, (const uint8_t*)w, (const uint8_t*)xq, y, m, (int)n,
                                        (int)k, stream));
}

plm_status gemm_ws_common(int fmt, const void* w, const void* xq, float* y, int64_t m, int64_t n,
                          int64_t k, void* ws, size_t ws_bytes, cudaStream_t stream) {
    plm_status s = check_matmul(w, xq, y, m, n, k, kMaxIndex);
    if (s != PLM_OK) return s;
    if (m * n > (int64_t)1 << 40) return PLM_ERR_INVALID_ARG;
    const size_t need = plm::gemm_workspace_need(fmt, m, (int)k);
    if (need > 0 && (!ws || ws_bytes < need)) return PLM_ERR_INVALID_ARG;
    if (ws && !aligned(ws, 256)) return PLM_ERR_MISALIGNED;
    if (!plm::gemv_supported(fmt, (int)k)) return PLM_ERR_UNSUPPORTED;
    return cuda_status(plm::launch_gemm_ws(fmt, (const uint8_t*)w, (const uint8_t*)xq, y, m, (int)n, (int)k,
                                           ws, ws_bytes, stream));
}

plm_status gemm_swiglu_common(const void* wg, const void* wu, const void* xq, float* h, int64_t m, int64_t n,
                              int64_t k, bool caller_ws, void* ws, size_t ws_bytes, cudaStream_t stream) {
    plm_status s = check_matmul(wg, xq, h, m, n, k, kMaxIndex);
    if (s != PLM_OK) return s;
    s = check_matmul(wu, xq, h, m, n, k, kMaxIndex);
    if (s != PLM_OK) return s;
    if (m * n > (int64_t)1 << 40) return PLM_ERR_INVALID_ARG;
    if (caller_ws) {
        const size_t need = plm::gemm_swiglu_workspace_min(m, (int)n, (int)k);
        if (need > 0 && (!ws || ws_bytes < need)) return PLM_ERR_INVALID_ARG;
        if (ws && !aligned(ws, 256)) return PLM_ERR_MISALIGNED;
    }
    if (!plm::gemv_supported(4, (int)k)) return PLM_ERR_UNSUPPORTED;
    const uint8_t *g8 = (const uint8_t*)wg, *u8 = (const uint8_t*)wu, *x8 = (const uint8_t*)xq;
    return cuda_status(caller_ws ? plm::launch_gemm_q4K_swiglu_ws(g8, u8, x8, h, m, (int)n, (int)k, ws, ws_bytes, stream)
                                 : plm::launch_gemm_q4K_swiglu(g8, u8, x8, h, m, (int)n, (int)k, stream));
}

plm_status subdots_common(int fmt, const void* w, const void* xq, int32_t* out, int64_t m,
                          int64_t n, int64_t k, cudaStream_t stream) {
    plm_status s = check_matmul(w, xq, out, m, n, k, plm::GEMV_MAX_M);
    if (s != PLM_OK) return s;
    if (!plm::gemv_supported(fmt, (int)k)) return PLM_ERR_UNSUPPORTED;
    return cuda_status(plm::launch_subdots(fmt, (const uint8_t*)w, (const uint8_t*)xq, out, (int)m,
                                           (int)n, (int)k, stream));
}

size_t x16_size(int fmt, int64_t n, int64_t k) {
    if (n <= 0 || k <= 0 || k % plm::QK != 0 || n > kMaxIndex || k > kMaxIndex) return 0;
    if (((n + 15) / 16) * (k / plm::QK) > kMaxIndex) return 0;
    return plm::x16_bytes(fmt, n, (int)k);
}

plm_status x16_repack(int fmt, const void* w, void* w_x16, int64_t n, int64_t k, cudaStream_t stream) {
    if (!w || !w_x16) return PLM_ERR_INVALID_ARG;
    if (x16_size(fmt, n, k) == 0) return PLM_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(w_x16, 16)) return PLM_ERR_MISALIGNED;
    return cuda_status(plm::launch_repack_x16(fmt, (const uint8_t*)w, (uint8_t*)w_x16, (int)n, (int)k, stream));
}

plm_status x16_gemv(int fmt, const void* w_x16, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                    cudaStream_t stream) {
    plm_status s = check_matmul(w_x16, xq, y, m, n, k, plm::GEMV_MAX_M);
    if (s != PLM_OK) return s;
    if (x16_size(fmt, n, k) == 0) return PLM_ERR_INVALID_ARG;
    return cuda_status(plm::launch_gemv_x16(fmt, (const uint8_t*)w_x16, (const uint8_t*)xq, y, (int)m, (int)n,
                                            (int)k, stream));
}

}  // namespace

extern "C" {

int plm_abi_version(void) { return PLM_ABI_VERSION; }

int plm_set_overlap(int mode) {
    if (mode < PLM_OVERLAP_OFF || mode > PLM_OVERLAP_PREFETCH) return -PLM_ERR_INVALID_ARG;
    return plm::g_overlap.exchange(mode);
}

const char* plm_status_string(int status) {
    switch (status) {
        case PLM_OK: return "ok";
        case PLM_ERR_INVALID_ARG: return "invalid argument";
        case PLM_ERR_MISALIGNED: return "misaligned pointer";
        case PLM_ERR_UNSUPPORTED: return "unsupported size";
        case PLM_ERR_CUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

int plm_last_cuda_error(void) { return g_last_cuda_error; }

plm_status plm_device_fault(uint32_t* code, int clear) {
    if (!code) return PLM_ERR_INVALID_ARG;
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, plm::g_plm_fault, sizeof v);
    if (e != cudaSuccess) return cuda_status(e);
    *code = v;
    if (clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(plm::g_plm_fault, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return PLM_OK;
}

plm_status plm_quantize_q8K(const float* x, void* xq, int64_t m, int64_t k, cudaStream_t stream) {
    if (!x || !xq) return PLM_ERR_INVALID_ARG;
    if (m <= 0 || k <= 0 || k % plm::QK != 0) return PLM_ERR_INVALID_ARG;
    if (m > kMaxIndex || k > kMaxIndex || m * (k / plm::QK) > kMaxIndex) return PLM_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 4)) return PLM_ERR_MISALIGNED;
    return cuda_status(plm::launch_quantize_q8K(x, (uint8_t*)xq, m, k, stream));
}

plm_status plm_gemv_q4K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemv_common(4, w, xq, y, m, n, k, stream);
}

plm_status plm_gemv_q6K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemv_common(6, w, xq, y, m, n, k, stream);
}

plm_status plm_gemv_q4K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream) {
    return grouped_common(4, problems, count, m, stream);
}

plm_status plm_gemv_q6K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream) {
    return grouped_common(6, problems, count, m, stream);
}

plm_status plm_gemv_q2K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemv_common(2, w, xq, y, m, n, k, stream);
}

plm_status plm_gemv_q2K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream) {
    return grouped_common(2, problems, count, m, stream);
}

plm_status plm_gemm_q2K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemm_common(2, w, xq, y, m, n, k, stream);
}

plm_status plm_gemm_q2K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return gemm_ws_common(2, w, xq, y, m, n, k, workspace, workspace_bytes, stream);
}

plm_status plm_subdots_q2K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream) {
    return subdots_common(2, w, xq, out, m, n, k, stream);
}

plm_status plm_gemv_q3K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemv_common(3, w, xq, y, m, n, k, stream);
}

plm_status plm_gemv_q3K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream) {
    return grouped_common(3, problems, count, m, stream);
}

plm_status plm_gemm_q3K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemm_common(3, w, xq, y, m, n, k, stream);
}

plm_status plm_gemm_q3K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return gemm_ws_common(3, w, xq, y, m, n, k, workspace, workspace_bytes, stream);
}

plm_status plm_subdots_q3K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream) {
    return subdots_common(3, w, xq, out, m, n, k, stream);
}

plm_status plm_gemv_q5K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemv_common(5, w, xq, y, m, n, k, stream);
}

plm_status plm_gemv_q5K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream) {
    return grouped_common(5, problems, count, m, stream);
}

plm_status plm_gemm_q5K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemm_common(5, w, xq, y, m, n, k, stream);
}

plm_status plm_gemm_q5K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return gemm_ws_common(5, w, xq, y, m, n, k, workspace, workspace_bytes, stream);
}

plm_status plm_subdots_q5K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream) {
    return subdots_common(5, w, xq, out, m, n, k, stream);
}

plm_status plm_gemm_q4K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemm_common(4, w, xq, y, m, n, k, stream);
}

plm_status plm_gemm_q6K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream) {
    return gemm_common(6, w, xq, y, m, n, k, stream);
}

size_t plm_gemm_workspace_size_split(int fmt, int64_t m, int64_t n, int64_t k) {
    if (fmt < 2 || fmt > 6 || m <= 0 || n <= 0 || k <= 0 || k % plm::QK != 0 || k > kMaxIndex || n > kMaxIndex ||
        m * n > (int64_t)1 << 40)
        return 0;
    return plm::gemm_workspace_need_split(fmt, m, (int)n, (int)k);
}

size_t plm_gemm_swiglu_workspace_size(int64_t m, int64_t n, int64_t k) {
    if (m <= 0 || n <= 0 || k <= 0 || k % plm::QK != 0 || k > kMaxIndex || n > kMaxIndex || m * n > (int64_t)1 << 40)
        return 0;
    return plm::gemm_swiglu_workspace_need(m, (int)n, (int)k);
}

size_t plm_gemm_workspace_size(int fmt, int64_t m, int64_t k) {
    if (fmt < 2 || fmt > 6 || m <= 0 || k <= 0 || k % plm::QK != 0 || k > kMaxIndex) return 0;
    return plm::gemm_workspace_need(fmt, m, (int)k);
}

plm_status plm_gemm_q4K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return gemm_ws_common(4, w, xq, y, m, n, k, workspace, workspace_bytes, stream);
}

plm_status plm_gemm_q6K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return gemm_ws_common(6, w, xq, y, m, n, k, workspace, workspace_bytes, stream);
}

plm_status plm_gemm_q4K_noalloc(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                                cudaStream_t stream) {
    plm_status s = check_matmul(w, xq, y, m, n, k, kMaxIndex);
    if (s != PLM_OK) return s;
    if (m * n > (int64_t)1 << 40) return PLM_ERR_INVALID_ARG;
    if (!plm::gemm_noalloc_fits(m, (int)k)) return PLM_ERR_UNSUPPORTED;   // beyond the fixed array
    if (!plm::gemv_supported(4, (int)k)) return PLM_ERR_UNSUPPORTED;
    return cuda_status(plm::launch_gemm_q4K_noalloc((const uint8_t*)w, (const uint8_t*)xq, y, m, (int)n, (int)k,
                                                    stream));
}

size_t plm_q4K_x16_size(int64_t n, int64_t k) { return x16_size(4, n, k); }
size_t plm_q6K_x16_size(int64_t n, int64_t k) { return x16_size(6, n, k); }

plm_status plm_q4K_to_x16(const void* w, void* w_x16, int64_t n, int64_t k, cudaStream_t stream) {
    return x16_repack(4, w, w_x16, n, k, stream);
}
plm_status plm_q6K_to_x16(const void* w, void* w_x16, int64_t n, int64_t k, cudaStream_t stream) {
    return x16_repack(6, w, w_x16, n, k, stream);
}

plm_status plm_gemv_q4K_x16(const void* w_x16, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                            cudaStream_t stream) {
    return x16_gemv(4, w_x16, xq, y, m, n, k, stream);
}
plm_status plm_gemv_q6K_x16(const void* w_x16, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                            cudaStream_t stream) {
    return x16_gemv(6, w_x16, xq, y, m, n, k, stream);
}

plm_status plm_quantize_gemv_q4K(const void* w, const float* x, float* y, int64_t m, int64_t n, int64_t k,
                                 cudaStream_t stream) {
    const plm_qgemv_problem p{w, x, y, n, k};
    return qgemv_common(&p, 1, m, stream);
}

plm_status plm_quantize_gemv_q4K_grouped(const plm_qgemv_problem* problems, int64_t count, int64_t m,
                                         cudaStream_t stream) {
    return qgemv_common(problems, count, m, stream);
}

plm_status plm_gemv_q4K_swiglu(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                               int64_t n, int64_t k, cudaStream_t stream) {
    const plm_swiglu_problem p{w_gate, w_up, xq, h, n, k};
    return swiglu_common(&p, 1, m, stream);
}

plm_status plm_gemm_q4K_swiglu(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                               int64_t n, int64_t k, cudaStream_t stream) {
    return gemm_swiglu_common(w_gate, w_up, xq, h, m, n, k, false, nullptr, 0, stream);
}

plm_status plm_gemm_q4K_swiglu_ws(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                                  int64_t n, int64_t k, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    return gemm_swiglu_common(w_gate, w_up, xq, h, m, n, k, true, workspace, workspace_bytes, stream);
}

plm_status plm_gemv_q4K_swiglu_grouped(const plm_swiglu_problem* problems, int64_t count, int64_t m,
                                       cudaStream_t stream) {
    return swiglu_common(problems, count, m, stream);
}

plm_status plm_subdots_q4K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n,
                           int64_t k, cudaStream_t stream) {
    return subdots_common(4, w, xq, out, m, n, k, stream);
}

plm_status plm_subdots_q6K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n,
                           int64_t k, cudaStream_t stream) {
    return subdots_common(6, w, xq, out, m, n, k, stream);
}

}  // extern "C"
