"""GB300 (sm_103a) packed K-quant matmul: q8_K activation quantization and
q2_K .. q6_K decode GEMV and prefill GEMM behind a C ABI (include/plm.h)."""
from .plm import (  # noqa: F401
    PlmError, load, library_path, plm_abi_version, plm_set_overlap,
    PLM_OVERLAP_OFF, PLM_OVERLAP_LAUNCH, PLM_OVERLAP_PREFETCH, plm_device_fault, plm_selftest_bounded_wait, plm_probe_mma_rates,
    plm_probe_tcgen05_rate, plm_quantize_q8K,
    plm_gemv_q4K, plm_gemv_q6K, plm_gemv_q4K_grouped, plm_gemv_q6K_grouped, plm_gemm_q4K, plm_gemm_q6K, plm_gemm_q4K_noalloc, plm_gemm_q4K_ws, plm_gemm_q6K_ws, plm_gemm_workspace_size, plm_gemm_workspace_size_split,
    plm_subdots_q4K, plm_subdots_q6K, plm_quantize_gemv_q4K, plm_quantize_gemv_q4K_grouped,
    plm_gemv_q4K_swiglu, plm_gemv_q4K_swiglu_grouped, plm_gemm_q4K_swiglu, plm_gemm_q4K_swiglu_ws,
    plm_gemm_swiglu_workspace_size,
    plm_gemv_q5K, plm_gemv_q5K_grouped, plm_gemm_q5K, plm_gemm_q5K_ws, plm_subdots_q5K, Q5K_BYTES,
    plm_gemv_q2K, plm_gemv_q2K_grouped, plm_gemm_q2K, plm_gemm_q2K_ws, plm_subdots_q2K, Q2K_BYTES,
    plm_gemv_q3K, plm_gemv_q3K_grouped, plm_gemm_q3K, plm_gemm_q3K_ws, plm_subdots_q3K, Q3K_BYTES,
    plm_q4K_x16_size, plm_q4K_to_x16, plm_gemv_q4K_x16, plm_q6K_x16_size, plm_q6K_to_x16, plm_gemv_q6K_x16,
    QK, Q4K_BYTES, Q6K_BYTES, Q8K_BYTES, GEMV_MAX_M,
)
