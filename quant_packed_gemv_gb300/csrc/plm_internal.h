// Host-side declarations shared by the plm translation units.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace plm {

// Number of SMs of the current device (queried per call; no cached state).
int num_sms();

// Early launch of the library's kernels (plm_set_overlap): 0 plain stream
// order; 1 a kernel may be scheduled while the kernel before it on the stream
// is still running and waits for it (griddepcontrol.wait) before its first
// memory access; 2 as 1, and a GEMV may copy weight bytes before that wait.
int overlap_mode();

// Launches kernel k, marked for early launch when overlap_mode() >= 1 (the
// kernel must then wait before touching memory that earlier work writes).
template <typename... P, typename... A>
inline cudaError_t launch_kernel(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 A&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = overlap_mode() >= 1 ? 1 : 0;
    return cudaLaunchKernelEx(&lc, k, std::forward<A>(args)...);
}

// The same with thread-block clusters of (1, 1, cz) CTAs along the grid's z.
template <typename... P, typename... A>
inline cudaError_t launch_kernel_cluster(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                         unsigned cz, A&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = cz;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = overlap_mode() >= 1 ? 2 : 1;
    return cudaLaunchKernelEx(&lc, k, std::forward<A>(args)...);
}

// Clusters of (1, 1, cz) CTAs of kernel k with this block and shared memory
// that the GPU can hold at once (0: none; the launch would fail).
template <typename... P>
inline int max_active_clusters(void (*k)(P...), dim3 grid, dim3 block, size_t smem, unsigned cz) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = cz;
    lc.attrs = at;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)k, &lc) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Device address of the library's fault word on the current device (set by a
// kernel whose bounded wait ran out), or nullptr if it cannot be resolved.
unsigned* fault_word();

cudaError_t launch_quantize_q8K(const float* x, uint8_t* xq, long long m, long long k,
                                cudaStream_t stream);

// False when one activation row of length k does not fit a CTA's shared memory.
bool gemv_supported(int fmt, int k);

// GEMV for 1 <= m <= 8 (q4_K: fmt = 4, q6_K: fmt = 6).
cudaError_t launch_gemv(int fmt, const uint8_t* w, const uint8_t* xq, float* y,
                        int m, int n, int k, cudaStream_t stream);

// A group of independent GEMVs sharing m, in one launch per 256 problems.
struct GroupItem {
    const uint8_t* w;
    const uint8_t* xq;
    float* y;
    int n, k;
    const uint8_t* w2 = nullptr;   // gate/up pairs: the up matrix
};
cudaError_t launch_gemv_grouped(int fmt, const GroupItem* items, int count, int m, cudaStream_t stream);

// Fused quantize + q4_K GEMV on f32 activations (GroupItem::xq holds the
// f32 activation pointer), one launch per 256 problems.
cudaError_t launch_quantize_gemv_q4K(const GroupItem* items, int count, int m, cudaStream_t stream);

// q4_K gate/up pairs with the SwiGLU epilogue (GroupItem::w = gate, w2 = up).
cudaError_t launch_gemv_q4K_swiglu(const GroupItem* items, int count, int m, cudaStream_t stream);

// Sub-block integer dots through the GEMV's lane decode (1 <= m <= 8).
cudaError_t launch_subdots(int fmt, const uint8_t* w, const uint8_t* xq, int32_t* out,
                           int m, int n, int k, cudaStream_t stream);

// Prefill GEMM, any m >= 1.  The _ws form uses the caller's workspace
// (gemm_workspace_need bytes, 256-byte aligned); the plain form needs none
// (the kernel widens the activation codes itself).
cudaError_t launch_gemm(int fmt, const uint8_t* w, const uint8_t* xq, float* y,
                        long long m, int n, int k, cudaStream_t stream);
cudaError_t launch_gemm_ws(int fmt, const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                           void* ws, size_t ws_bytes, cudaStream_t stream);
size_t gemm_workspace_need(int fmt, long long m, int k);

// q4_K gate/up pair with the SwiGLU epilogue, any m; the _ws form takes the
// up matrix's output, then a GEMM workspace: gemm_swiglu_workspace_need(m, n,
// k) bytes splits K where that pays, gemm_swiglu_workspace_min is the least
// it accepts (unsplit).
size_t gemm_swiglu_workspace_need(long long m, int n, int k);
size_t gemm_swiglu_workspace_min(long long m, int n, int k);
cudaError_t launch_gemm_q4K_swiglu(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* xq, float* h,
                                   long long m, int n, int k, cudaStream_t stream);
cudaError_t launch_gemm_q4K_swiglu_ws(const uint8_t* w_gate, const uint8_t* w_up, const uint8_t* xq, float* h,
                                      long long m, int n, int k, void* ws, size_t ws_bytes, cudaStream_t stream);
// The same plus the partial sums of a K split (used when the output tiles
// alone would leave most SMs idle); the _ws form splits K only when given this.
size_t gemm_workspace_need_split(int fmt, long long m, int n, int k);

// Allocation-free q4_K GEMM: the workspace is a fixed device array inside the
// library (PLM_NOALLOC_WORKSPACE_BYTES).
bool gemm_noalloc_fits(long long m, int k);
cudaError_t launch_gemm_q4K_noalloc(const uint8_t* w, const uint8_t* xq, float* y, long long m, int n, int k,
                                    cudaStream_t stream);

// Row-interleaved q4_K / q6_K layouts "x16" (tiles of 16 rows per 256-weight block):
// bytes of the repacked matrix, the repack, and the tensor-core decode GEMV
// over it (1 <= m <= 8).
size_t x16_bytes(int fmt, long long n, int k);   // fmt 4 (q4_K) or 6 (q6_K)
cudaError_t launch_repack_x16(int fmt, const uint8_t* w, uint8_t* out, int n, int k, cudaStream_t stream);
cudaError_t launch_gemv_x16(int fmt, const uint8_t* w, const uint8_t* xq, float* y, int m, int n, int k,
                            cudaStream_t stream);

}  // namespace plm
