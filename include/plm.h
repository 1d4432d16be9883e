/*
 * plm -- packed K-quant matmul (gemm_quant) for GB300 (sm_103a).
 *
 * The operation is the packed-weight matmul of the PocketLLM pages ("What it
 * runs": q4_k / q6_k weights decoded inside the kernel and never widened;
 * "Current status", row "src/ -- the C++ engine": activations quantized to
 * int8 one 256-element block at a time, the q6_K output head summed in
 * int32).  The byte formats are the public GGML K-quant blocks those pages
 * name:
 *
 *   q4_K (144 B per 256 weights): f16 d, f16 dmin, u8 scales[12] (eight
 *        6-bit scale/min pairs), u8 qs[128] (4-bit codes; each 64-weight
 *        chunk keeps its first 32 weights in the low nibbles, the next 32 in
 *        the high nibbles).  weight = d*sc_j*q - dmin*m_j.
 *   q6_K (210 B per 256 weights): u8 ql[128], u8 qh[64], i8 scales[16]
 *        (one per 16 weights), f16 d.  weight = d*sc*(q6 - 32).
 *   q8_K (292 B per 256 activations): f32 d, i8 qs[256], i16 bsums[16].
 *
 * Shapes and layouts (all row-major, no padding):
 *   m  activation rows, n weight (output) rows, k reduction length,
 *      k a positive multiple of 256, nb = k/256.
 *   x  f32  [m][k]
 *   xq q8_K [m][nb]      (m*nb*292 bytes)
 *   w  q4_K [n][nb] or q6_K [n][nb]   (n*nb*144 or n*nb*210 bytes)
 *   y  f32  [m][n]       y[i][r] = sum over k of x_hat[i][.] * w_hat[r][.]
 *
 * Ownership and ordering: every pointer is a DEVICE pointer owned by the
 * caller.  The library never synchronizes and allocates nothing; the _ws
 * forms use a workspace the caller passes.  Each call
 * enqueues its work on `stream` (0 = the legacy default stream) and returns
 * at once; results are visible to later work on that stream.  y is
 * overwritten, never accumulated into.  Calls on different streams that
 * write the same buffers race.
 *
 * Errors: arguments are checked on the host before anything is enqueued;
 * a rejected call enqueues nothing.  PLM_ERR_INVALID_ARG: null pointer,
 * m, n <= 0, k <= 0 or k % 256 != 0, GEMV with m > 8, sizes past int32
 * indexing.  PLM_ERR_MISALIGNED: a pointer below the alignment its entry
 * point states.  PLM_ERR_CUDA: the launch itself failed (the CUDA error code
 * is then available from plm_last_cuda_error on the calling thread).
 * Faults inside kernels are never used to report errors.
 */
#ifndef PLM_H
#define PLM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PLM_ABI_VERSION 1

typedef enum {
    PLM_OK = 0,
    PLM_ERR_INVALID_ARG = 1,
    PLM_ERR_MISALIGNED = 2,
    PLM_ERR_UNSUPPORTED = 3,
    PLM_ERR_CUDA = 4
} plm_status;

/* ABI version of the loaded library (PLM_ABI_VERSION at build time). */
int plm_abi_version(void);

/*
 * Early launch (no counterpart on the pages; a GB300 scheduling feature).
 * Process-wide mode for every kernel launched after the call:
 *   PLM_OVERLAP_OFF       plain stream order: a kernel starts when the work
 *                         before it on the stream has finished.
 *   PLM_OVERLAP_LAUNCH    (default) kernels are launched with programmatic
 *                         stream serialization: a kernel may be scheduled
 *                         while the kernel before it is still running, and
 *                         waits for that kernel and its memory writes before
 *                         its own first memory access.  Results are the same
 *                         as in plain order; the launch latency is hidden.
 *   PLM_OVERLAP_PREFETCH  as PLM_OVERLAP_LAUNCH, and a GEMV may start copying
 *                         its weight bytes before that wait (activations are
 *                         read and y written only after it), so its weight
 *                         stream overlaps the tail of the kernel before it.
 *                         The caller guarantees that no kernel issued earlier
 *                         on the same stream writes the weight bytes of a
 *                         GEMV call (weights are immutable once loaded);
 *                         otherwise the GEMV may read stale weights.
 * Returns the previous mode, or -PLM_ERR_INVALID_ARG (mode unchanged) for
 * any other value.  Safe to call from any thread; launches already enqueued
 * keep the mode they were issued with.
 */
#define PLM_OVERLAP_OFF 0
#define PLM_OVERLAP_LAUNCH 1
#define PLM_OVERLAP_PREFETCH 2
int plm_set_overlap(int mode);

/* Static, NUL-terminated name of a status code; "unknown status" otherwise. */
const char* plm_status_string(int status);

/* cudaError_t of the last PLM_ERR_CUDA returned on the calling thread
 * (cudaSuccess if none). */
int plm_last_cuda_error(void);

/*
 * Diagnostic: the device fault word of the current device.  Kernels that
 * stream through asynchronous copies bound every wait; a wait that runs out
 * sets bit 0 here and the kernel stops (its outputs are then incomplete).
 * *code receives the word; clear != 0 resets it.  Unlike the compute entry
 * points this call synchronizes with the device (it copies one word).
 */
plm_status plm_device_fault(uint32_t* code, int clear);

/*
 * Failure-detection self-test (no counterpart on the pages; it checks the
 * library's own error path).  Launches one warp on `stream` that waits on a
 * shared-memory mbarrier with the bounded wait every streaming kernel uses,
 * limited to `rounds` rounds of at most 20 microseconds each (1 <= rounds <=
 * 65536, else PLM_ERR_INVALID_ARG and nothing is launched).  complete != 0:
 * the barrier's one arrival is made before the wait, which then ends at once
 * and leaves the fault word alone.  complete == 0: nothing arrives and no
 * copy is in flight, so the wait runs out, the kernel sets bit 0 of the
 * device fault word (read it with plm_device_fault) and returns; the device
 * stays usable.  Allocates nothing, does not synchronize.  PLM_ERR_CUDA if
 * the launch failed.
 */
plm_status plm_selftest_bounded_wait(uint32_t rounds, int complete, cudaStream_t stream);

/*
 * Diagnostic (the pages have no counterpart): measured throughput of the
 * warp-level tensor instructions mma.sync m16n8k32 s8 (*s8_tops, TOPS) and
 * mma.sync m16n8k16 f16 with f32 accumulation (*f16_tflops, TFLOPS) on the
 * current device, from register-only loops on the legacy default stream.
 * Context only: tcgen05 on sm_103a has no int8 kind, and both legacy rates
 * are far below the tcgen05 f16 dense rate.  Synchronizes; allocates
 * nothing.
 */
plm_status plm_probe_mma_rates(double* s8_tops, double* f16_tflops);

/*
 * Diagnostic (the pages have no counterpart): the tcgen05 MMA the prefill
 * GEMM issues (kind::f16, M = 128, N = 128, K = 16, A from tensor memory, B
 * from shared memory, zero operands), streamed by one thread with a commit
 * every four MMAs.
 *   *cycles_per_mma      : SM cycles per MMA, one CTA;
 *   *cycles_per_mma_wait : the same with an mbarrier wait on an already
 *                          completed phase after each commit (what a wait
 *                          in the MMA-issuing thread costs the tensor pipe);
 *   *tflops              : the first pattern on one CTA per SM (dense rate on
 *                          zero operands: context, not a roofline peak).
 * Synchronizes; allocates nothing (a static device array holds the cycle
 * counts).  PLM_ERR_CUDA if a launch failed; a wait that runs out sets bit 1
 * of plm_device_fault.
 */
plm_status plm_probe_tcgen05_rate(double* cycles_per_mma, double* cycles_per_mma_wait, double* tflops);

/*
 * q8_K activation quantization ("Current status" row "src/": activations
 * quantized to int8 the llama.cpp way, one 256-element block per task).
 * Per 256-element chunk of each row of x: the signed value `max` of largest
 * magnitude (first occurrence on ties), iscale = -128/max, code =
 * min(127, round-half-even(iscale*x)), d = 1/iscale, bsums[g] = sum of codes
 * 16g..16g+15; an all-zero chunk gives d = 0 and zero codes and sums.
 * Bit-exact with that scalar rule.
 *   x  : f32 [m][k], 16-byte aligned.       xq : q8_K [m][k/256], 4-byte aligned.
 */
plm_status plm_quantize_q8K(const float* x, void* xq, int64_t m, int64_t k,
                            cudaStream_t stream);

/*
 * Decode GEMV, y = W . x for m = 1..8 activation rows ("What it runs":
 * packed weights decoded in the kernel; the weight stream is read once for
 * all m rows, as the pages' 8-row activation tile does).  Integer sub-block
 * dots are exact; the f32 result is within 1e-4 of sum_k |w_hat * x_hat|.
 * The result for activation row i does not depend on m.
 *   w  : q4_K [n][k/256], 16-byte aligned.  xq : q8_K [m][k/256], 4-byte aligned.
 *   y  : f32 [m][n], 4-byte aligned.        1 <= m <= 8.
 */
plm_status plm_gemv_q4K(const void* w, const void* xq, float* y,
                        int64_t m, int64_t n, int64_t k, cudaStream_t stream);

/* q6_K decode GEMV (the output head path of "Current status" row "src/",
 * summed in int32).  Same contract as plm_gemv_q4K; w is q6_K
 * [n][k/256] and must be 16-byte aligned. */
plm_status plm_gemv_q6K(const void* w, const void* xq, float* y,
                        int64_t m, int64_t n, int64_t k, cudaStream_t stream);

/*
 * A group of independent decode GEMVs in one launch: problem j computes
 * y_j = W_j . x_j exactly as plm_gemv_q4K(w_j, xq_j, y_j, m, n_j, k_j) would
 * (same bits), for matrices that do not depend on one another: the q/k/v or
 * gate/up projections of a layer kept as separate tensors, the experts of a
 * mixture-of-experts layer, or a whole set of decode matrices.
 *   problems : HOST array of `count` descriptors, read during the call only.
 *   m        : activation rows of every problem, 1 <= m <= 8.
 * Each descriptor obeys the single-GEMV rules (alignment, k % 256 == 0); the
 * call checks all of them before launching anything.  Distinct problems may
 * share w or xq but must not share y.
 */
typedef struct {
    const void* w;    /* q4_K or q6_K [n][k/256] */
    const void* xq;   /* q8_K [m][k/256] */
    float* y;         /* f32 [m][n] */
    int64_t n;
    int64_t k;
} plm_gemv_problem;

plm_status plm_gemv_q4K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream);
plm_status plm_gemv_q6K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream);

/*
 * q2_K and q3_K, the lowest rungs of the pages' K-quant width ladder
 * (PocketLLM README, "What it runs": q2_k, q3_k and q5_k join q4_k and q6_k
 * as formats the engine decodes).  Public GGML layouts, sixteen 16-weight
 * groups per 256 weights; group g holds weights 16g..16g+15 and, with
 * h = g/8, j = (g%8)/2, p = g%2, its 2-bit codes are bits 2j..2j+1 of
 * qs[32h + 16p + l]:
 *   q2_K (84 bytes): u8 scales[16] (low nibble scale sc_g, high nibble min
 *        m_g), u8 qs[64], f16 d, f16 dmin; weight = d * sc_g * q - dmin * m_g.
 *   q3_K (110 bytes): u8 hmask[32] (bit 4h + j of hmask[16p + l] is the
 *        weight's third bit), u8 qs[64], u8 scales[12] (6-bit s_g: low four
 *        bits from scales[g % 8], nibble g / 8; top two from scales[8 + g % 4],
 *        bits 2(g/4)..), f16 d; code q3 = q - 4 when the third bit is clear,
 *        weight = d * (s_g - 32) * q3.
 * Blocks are 4-byte (q2_K) / 2-byte (q3_K) aligned inside a row; w must be
 * 16-byte aligned.  Same contracts and errors as the q6_K entry points; the
 * sub-dot export writes the int32 16-weight group dots, [m][n][k/16].  The
 * GEMM entry points run on the tensor cores for m >= 9 when a row of blocks
 * is a multiple of 16 bytes (q2_K: k/256 % 4 == 0; q3_K: k/256 % 8 == 0):
 * operands sc_g * q (q2_K, with the mins as a second contraction against the
 * bsums) and (s_g - 32) * (q3 + 4) (q3_K, with the -4 (s_g - 32) bsum part as
 * the second contraction), all exact in f16.  Other shapes run the decode
 * GEMV eight activation rows at a time (no workspace, size 0).
 */
plm_status plm_gemv_q2K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemv_q2K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream);
plm_status plm_gemm_q2K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemm_q2K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
plm_status plm_subdots_q2K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream);
plm_status plm_gemv_q3K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemv_q3K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream);
plm_status plm_gemm_q3K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemm_q3K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
plm_status plm_subdots_q3K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream);

/*
 * q5_K, the next rung of the pages' K-quant width ladder (PocketLLM README,
 * "What it runs": q2_k, q3_k, q5_k join q4_k and q6_k as formats the engine
 * decodes).  Block (176 bytes per 256 weights, the public GGML layout): f16 d,
 * f16 dmin, u8 scales[12] (q4_K's eight 6-bit (scale, min) pairs), u8 qh[32],
 * u8 qs[128]; weight 64c + l (l < 32) = low nibble of qs[32c + l] + 16 * bit
 * 2c of qh[l], weight 64c + 32 + l = high nibble + 16 * bit 2c + 1;
 * value d * sc_j * q5 - dmin * m_j.  Same contracts, layouts, alignment and
 * errors as the q4_K entry points (w 16-byte aligned); the sub-dot export
 * writes int32 [m][n][k/32] like q4_K's.
 */
plm_status plm_gemv_q5K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemv_q5K_grouped(const plm_gemv_problem* problems, int64_t count, int64_t m,
                                cudaStream_t stream);
plm_status plm_gemm_q5K(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                        cudaStream_t stream);
plm_status plm_gemm_q5K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
plm_status plm_subdots_q5K(const void* w, const void* xq, int32_t* out, int64_t m, int64_t n, int64_t k,
                           cudaStream_t stream);

/*
 * Fused q8_K producer + decode GEMV (q4_K), y = W . x for 1 <= m <= 8, on
 * f32 activations.  PocketLLM (Korean README), "Current status" table, row
 * "src/": the packed matmul runs on int8 activations quantized per 256-value
 * block; here that quantization happens inside the GEMV launch.  Each CTA
 * quantizes the activation rows of the problems it covers with the same
 * arithmetic as plm_quantize_q8K (first-occurrence signed amax,
 * iscale = -128/max, round half to even, clamp at 127, d = 1/iscale), so y is
 * bit-identical to plm_quantize_q8K followed by plm_gemv_q4K, without the
 * q8_K round trip through memory or the second launch.
 *   x  device f32 [m][k], 16-byte aligned (else PLM_ERR_MISALIGNED);
 *   w, y as for plm_gemv_q4K.  No workspace, nothing allocated.
 *   x and y may also be pinned host memory that the device addresses
 *   directly (unified addressing): the kernel then reads x and writes y
 *   across the CPU-GPU link itself, with no copy call.
 * Errors as for plm_gemv_q4K.
 */
plm_status plm_quantize_gemv_q4K(const void* w, const float* x, float* y, int64_t m, int64_t n, int64_t k,
                                 cudaStream_t stream);

/* Grouped form: independent problems sharing m, f32 activations each. */
typedef struct {
    const void* w;    /* q4_K [n][k/256] */
    const float* x;   /* f32 [m][k], 16-byte aligned */
    float* y;         /* f32 [m][n] */
    int64_t n;
    int64_t k;
} plm_qgemv_problem;

plm_status plm_quantize_gemv_q4K_grouped(const plm_qgemv_problem* problems, int64_t count, int64_t m,
                                         cudaStream_t stream);

/*
 * Gate/up pair with the SwiGLU epilogue (q4_K), 1 <= m <= 8:
 *   h[i][r] = silu(g[i][r]) * u[i][r],  g = W_gate . x_i,  u = W_up . x_i,
 *   silu(g) = g / (1 + exp(-g)).
 * PocketLLM (Korean README), "Current status" table, row "src/": the decode
 * path's silu_mul step after the ffn gate and up projections.  Both weight
 * matrices stream in one launch; g and u are the same f32 values
 * plm_gemv_q4K produces for each matrix (same order), combined in f32 with
 * IEEE division and expf, so only the epilogue's rounding separates h from
 * silu applied to plm_gemv_q4K's outputs.
 *   w_gate, w_up  q4_K [n][k/256] each, 16-byte aligned; xq q8_K [m][k/256];
 *   h f32 [m][n].  Errors as for plm_gemv_q4K.
 */
plm_status plm_gemv_q4K_swiglu(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                               int64_t n, int64_t k, cudaStream_t stream);

typedef struct {
    const void* w_gate;   /* q4_K [n][k/256] */
    const void* w_up;     /* q4_K [n][k/256] */
    const void* xq;       /* q8_K [m][k/256] */
    float* h;             /* f32 [m][n] */
    int64_t n;
    int64_t k;
} plm_swiglu_problem;

plm_status plm_gemv_q4K_swiglu_grouped(const plm_swiglu_problem* problems, int64_t count, int64_t m,
                                       cudaStream_t stream);

/*
 * Prefill GEMM, y = X . W^T for any m >= 1 (intended for m = 512..2048).
 * For m >= 9, weight tiles are decoded into exact integer-valued f16
 * operands (q4_K: sc*q; q6_K: 16*hi*(q6-32) and lo*(q6-32) for sc = 16*hi
 * + lo, two contractions into one accumulator) and
 * contracted on the tensor cores (tcgen05, f32 accumulation in tensor
 * memory) against the activation codes as exact f16, one 256-weight block at
 * a time; the per-block scales are applied in f32.  These plain forms widen
 * the activation codes inside the GEMM kernel, straight from xq into shared
 * memory: they need no workspace and allocate nothing.  When the output
 * tiles alone would leave SMs idle (small m and n), they split K over a
 * thread-block cluster of up to eight CTAs per tile and rank 0 adds the
 * partial tiles from the others' shared memory in rank order (the same bits
 * every run; q6_K only where k/256 % 8 == 0, its other shapes do not split).  For
 * m <= 8 (and q2_K / q3_K shapes without the tensor-core path, see above)
 * they run the decode GEMV eight rows at a time.
 * Same buffers, layouts and tolerance as the GEMV; no limit on m.  A _ws
 * call that splits K the same way (given plm_gemm_workspace_size_split bytes,
 * at most eight splits) or does not split where the plain call does not
 * gives the same bits.
 */
plm_status plm_gemm_q4K(const void* w, const void* xq, float* y,
                        int64_t m, int64_t n, int64_t k, cudaStream_t stream);
plm_status plm_gemm_q6K(const void* w, const void* xq, float* y,
                        int64_t m, int64_t n, int64_t k, cudaStream_t stream);

/*
 * Gate/up pair with the SwiGLU epilogue for prefill (q4_K), any m >= 1:
 *   h[i][r] = silu(g[i][r]) * u[i][r],  g = W_gate . x_i,  u = W_up . x_i,
 * the same step as plm_gemv_q4K_swiglu (PocketLLM (Korean README), "Current
 * status" table, row "src/": silu_mul after the ffn gate and up projections)
 * at prefill sizes, h = silu(g) * u = g / (1 + e^-g) * u (IEEE division,
 * expf).  For m >= 9 the plain form runs the q4_K GEMM of the gate matrix
 * into h, then that of the up matrix, whose epilogue reads each element's g
 * back from h and writes silu(g) * u over it: no workspace, nothing
 * allocated.  The _ws form runs the two GEMMs (the up matrix's into the
 * workspace, K split when the workspace allows) and one elementwise pass;
 * where both split K alike (or neither does) they give the same bits.  For
 * m <= 8 both run
 * plm_gemv_q4K_swiglu eight rows at a time.
 *   w_gate, w_up  q4_K [n][k/256] each, 16-byte aligned; xq q8_K [m][k/256];
 *   h f32 [m][n], not overlapping the inputs.  The _ws form's workspace:
 *   plm_gemm_swiglu_workspace_size(m, n, k) bytes (K split where it pays)
 *   or at least m*n*4 rounded up to 256 plus plm_gemm_workspace_size(4, m, k)
 *   (unsplit), 256-byte aligned (null allowed when the size is 0).  Errors as
 *   for plm_gemm_q4K / plm_gemm_q4K_ws.
 */
plm_status plm_gemm_q4K_swiglu(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                               int64_t n, int64_t k, cudaStream_t stream);
plm_status plm_gemm_q4K_swiglu_ws(const void* w_gate, const void* w_up, const void* xq, float* h, int64_t m,
                                  int64_t n, int64_t k, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);
/* Workspace bytes of plm_gemm_q4K_swiglu_ws: m >= 9: m*n*4 (the up matrix's
 * output, rounded up to 256 bytes) plus plm_gemm_workspace_size_split(4, m,
 * n, k); 0 for m <= 8 and for invalid arguments. */
size_t plm_gemm_swiglu_workspace_size(int64_t m, int64_t n, int64_t k);

/* Workspace bytes plm_gemm_qNK_ws needs (fmt = N: 2, 3, 4, 5, 6; q2_K and
 * q3_K only on shapes with the tensor-core path, see above, else none) for m
 * activation rows of length k: for m >= 9, the codes
 * widened to f16 (2*m*k bytes) and, per activation row and 256-value block,
 * 48 bytes of side data (the bsums as f16 pairs and d), each part rounded up
 * to 256 bytes.  0 when none is needed, and for invalid arguments. */
size_t plm_gemm_workspace_size(int fmt, int64_t m, int64_t k);

/* Workspace that also holds the partial sums of a K split: when the output
 * tiles of an m x n problem alone would leave most SMs idle (small m, small
 * n), the tensor-core GEMM splits K over up to (SMs / tiles) CTAs per tile,
 * writes each split's f32 partial y into the workspace and adds the splits
 * in a fixed order (so the result does not depend on timing).  The _ws entry
 * points split K only when given at least this many bytes; with the smaller
 * plm_gemm_workspace_size they run unsplit.  0 for invalid arguments and when
 * no workspace is needed. */
size_t plm_gemm_workspace_size_split(int fmt, int64_t m, int64_t n, int64_t k);

/* The GEMM with a caller-owned device workspace of at least
 * plm_gemm_workspace_size bytes, 256-byte aligned (may be null when that
 * size is 0).  A pre-pass widens the activation codes into the workspace and
 * the GEMM kernel loads them by TMA; with plm_gemm_workspace_size_split
 * bytes K is split where the output tiles alone would leave SMs idle (the
 * faster choice for small m and n).  The workspace must not be used by other
 * work until the call's kernels have finished on `stream`.
 * PLM_ERR_INVALID_ARG if it is too small. */
plm_status plm_gemm_q4K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);
plm_status plm_gemm_q6K_ws(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Allocation-free q4_K GEMM through a fixed workspace.  No counterpart on
 * the PocketLLM pages: it is a library convenience.  It runs the workspace
 * form of the GEMM (plm_gemm_q4K_ws: pre-pass, TMA-loaded f16 activations,
 * no K split) with the workspace in a fixed device array inside this
 * library; results agree with plm_gemm_q4K, which needs no workspace at
 * all, bit for bit where that one does not split K either.  It is meant for callers that must not allocate device
 * memory while running, such as an engine whose memory is entirely claimed
 * by its own allocator at start-up, or a latency-critical loop that cannot
 * afford an allocation that might fail or wait.
 *   - Limit: the workspace of plm_gemm_workspace_size(4, m, k) (2*m*k bytes
 *     of f16 codes plus 48 bytes per 256-value block of activations, for
 *     m >= 9; smaller m needs none) must fit
 *     PLM_NOALLOC_WORKSPACE_BYTES; larger problems return
 *     PLM_ERR_UNSUPPORTED and enqueue nothing.
 *   - Calls no cudaMalloc, cudaFree or allocating routine.  Every device
 *     that loads the library holds the array until the process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture that includes this entry point.
 *   - All calls share the one array (it keeps the last call's contents, and
 *     each call rewrites the part it reads), so calls whose kernels may
 *     overlap on the GPU, e.g. on different streams, race: serialize them.
 *   - It never splits K (the array holds no split partial sums), so where
 *     plm_gemm_q4K_ws with the split workspace would split K -- few output
 *     tiles, i.e. small m and n -- it can be slower.
 *   - The array's device address is kept per device for the life of the
 *     process; do not call it across a cudaDeviceReset.
 */
#define PLM_NOALLOC_WORKSPACE_BYTES (32u << 20)
plm_status plm_gemm_q4K_noalloc(const void* w, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                                cudaStream_t stream);

/*
 * Row-interleaved q4_K layout "x16" and its tensor-core decode GEMV.
 * PocketLLM (Korean README), "Current status" table, row "src/": the packed
 * q4_K dot runs faster on a load-time repack of the weights (an 8-column
 * panel) with an 8-row activation tile.  Here the repack interleaves 16
 * weight rows per 256-weight block, the layout a warp-level tensor-core tile
 * reads with full 16-byte loads, and the m <= 8 activation rows form the
 * MMA's columns.  The layout holds the same bytes as the GGML q4_K blocks,
 * permuted in 16-byte units:
 *   rows are grouped in tiles of 16 (rows n .. 16*ceil(n/16) - 1 are zero
 *   blocks); the tile-block of tile T and block b (rows 16T .. 16T+15) is
 *   2304 contiguous bytes at ((T * (k/256)) + b) * 2304; inside it, bytes
 *   [0, 256) are the 16-byte headers (f16 d, f16 dmin, scales[12]) of the
 *   tile's rows in row order, and for j = 0..3 and L = 0..31 (g = L/4,
 *   t = L%4) bytes 256 + 512j + 16L .. +15 are qs[32t + 16(j%2) .. +15] of
 *   row 16T + g (j < 2) or row 16T + g + 8 (j >= 2).
 *
 * plm_q4K_x16_size: bytes of the x16 form of an n x k q4_K matrix
 *   (ceil(n/16) * (k/256) * 2304); 0 for invalid arguments.
 * plm_q4K_to_x16: writes that form of w (q4_K [n][k/256], device, 16-byte
 *   aligned) into w_x16 (device, plm_q4K_x16_size bytes, 16-byte aligned, not
 *   overlapping w).  Run once when the weights are loaded.  Under
 *   PLM_OVERLAP_PREFETCH, a GEMV that follows it on the same stream must not
 *   read w_x16 before it is written: synchronize (or use another mode) between
 *   the repack and the first GEMV.
 * plm_gemv_q4K_x16: y = W . x for 1 <= m <= 8 with W in the x16 form (n, k
 *   of the original matrix); xq and y as for plm_gemv_q4K.  Integer products
 *   are exact (f16 operands sc*q and q8 codes, f32 accumulation), the block
 *   terms d_x*(d*isum - dmin*msum) are formed in f32, and the result is within
 *   1e-4 of sum_k |w_hat * x_hat| per element.  The result for activation row
 *   i does not depend on m.  Errors as for plm_gemv_q4K.
 */
size_t plm_q4K_x16_size(int64_t n, int64_t k);
plm_status plm_q4K_to_x16(const void* w, void* w_x16, int64_t n, int64_t k, cudaStream_t stream);
plm_status plm_gemv_q4K_x16(const void* w_x16, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                            cudaStream_t stream);

/*
 * The x16 layout of q6_K (the output head, "Current status" row "src/":
 * summed in int32 because its sub-blocks overflow int16) and its tensor-core
 * decode GEMV.  Same bytes as the GGML q6_K blocks, rearranged in 4-byte
 * pieces: rows in tiles of 16 (rows n .. 16*ceil(n/16) - 1 zero); the
 * tile-block of tile T, block b is 3360 bytes at ((T * (k/256)) + b) * 3360:
 *   [0, 256)      the 16 int8 scales of row 16T + i at 16 i;
 *   [256, 288)    the f16 d of row 16T + i at 256 + 2 i;
 *   [288, 2336)   for j = 0..3, L = 0..31 (g = L/4, t = L%4): 16 bytes at
 *                 288 + 512 j + 16 L holding ql[64h + 16w + 4t .. +3] for
 *                 w = 0..3 (h = j % 2) of row 16T + g (j < 2) or 16T + g + 8;
 *   [2336, 3360)  for j = 0..1: 16 bytes at 2336 + 512 j + 16 L holding
 *                 qh[32h + 16s + 4t .. +3] for (h, s) = (0,0), (0,1), (1,0),
 *                 (1,1) of row 16T + g + 8 j.
 * plm_q6K_x16_size / plm_q6K_to_x16 / plm_gemv_q6K_x16: as the q4_K forms
 * (w q6_K [n][k/256], device, 16-byte aligned; 3360 bytes per tile-block).
 * The GEMV forms each 16-group's dot with (q6 - 32) codes exact in f16 and
 * applies the group's int8 scale to the exact integer result in f32, so
 * every int8 scale is exact; same tolerance, errors and m-independence as
 * plm_gemv_q4K_x16.
 */
size_t plm_q6K_x16_size(int64_t n, int64_t k);
plm_status plm_q6K_to_x16(const void* w, void* w_x16, int64_t n, int64_t k, cudaStream_t stream);
plm_status plm_gemv_q6K_x16(const void* w_x16, const void* xq, float* y, int64_t m, int64_t n, int64_t k,
                            cudaStream_t stream);

/*
 * Verification export: the integer sub-block dots computed by the same
 * device decode/dot code the GEMV uses.
 *   q4_K: out int32 [m][n][k/32],  out[i][r][8b+j]  = sum_{l<32} q * q8
 *         over sub-block j of block b.
 *   q6_K: out int32 [m][n][k/16],  out[i][r][16b+g] = sum_{l<16} (q6-32) * q8
 *         over group g of block b.
 *   Same alignment rules as the GEMV; out 4-byte aligned; 1 <= m <= 8.
 */
plm_status plm_subdots_q4K(const void* w, const void* xq, int32_t* out,
                           int64_t m, int64_t n, int64_t k, cudaStream_t stream);
plm_status plm_subdots_q6K(const void* w, const void* xq, int32_t* out,
                           int64_t m, int64_t n, int64_t k, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PLM_H */
