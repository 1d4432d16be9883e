"""Host-only checks of the C ABI: the library loads, exports every entry
point include/plm.h declares, and rejects bad arguments before any CUDA
call (no GPU needed; no kernel is launched by these tests)."""
import ctypes
import os
import re

import pytest

import quant_packed_gemv_gb300 as q
from quant_packed_gemv_gb300 import plm as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "plm.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(plm_[A-Za-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = q.load()
    names = declared_symbols()
    assert "plm_gemv_q4K" in names and "plm_quantize_q8K" in names and len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings():
    assert q.plm_abi_version() == 1
    lib = q.load()
    assert lib.plm_status_string(0) == b"ok"
    assert lib.plm_status_string(2) == b"misaligned pointer"
    assert lib.plm_status_string(99) == b"unknown status"
    assert lib.plm_last_cuda_error() == 0


def test_overlap_mode_setting():
    prev = q.plm_set_overlap(q.PLM_OVERLAP_OFF)
    try:
        assert prev == q.PLM_OVERLAP_LAUNCH   # the default; every test restores it
        assert q.plm_set_overlap(q.PLM_OVERLAP_PREFETCH) == q.PLM_OVERLAP_OFF
        assert q.plm_set_overlap(q.PLM_OVERLAP_LAUNCH) == q.PLM_OVERLAP_PREFETCH
        for bad in (3, -1, 1 << 20):
            with pytest.raises(q.PlmError):
                q.plm_set_overlap(bad)
        assert q.plm_set_overlap(q.PLM_OVERLAP_LAUNCH) == q.PLM_OVERLAP_LAUNCH
    finally:
        q.plm_set_overlap(prev)


A = 1 << 20  # a 16-byte aligned fake address; never dereferenced: every call below is rejected


@pytest.mark.parametrize("name", ["plm_gemv_q4K", "plm_gemv_q6K", "plm_gemm_q4K", "plm_gemm_q6K",
                                  "plm_subdots_q4K", "plm_subdots_q6K", "plm_quantize_gemv_q4K"])
def test_matmul_argument_checks(name):
    st = lambda *a: P.raw_status(name, *a)  # noqa: E731
    bad = P.PLM_ERR_INVALID_ARG
    assert st(None, A, A, 1, 8, 256, None) == bad
    assert st(A, None, A, 1, 8, 256, None) == bad
    assert st(A, A, None, 1, 8, 256, None) == bad
    assert st(A, A, A, 0, 8, 256, None) == bad
    assert st(A, A, A, 1, 0, 256, None) == bad
    assert st(A, A, A, 1, 8, 0, None) == bad
    assert st(A, A, A, 1, 8, 300, None) == bad
    assert st(A, A, A, -1, 8, 256, None) == bad
    assert st(A, A, A, 1, 1 << 40, 256, None) == bad
    assert st(A + 8, A, A, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED
    assert st(A, A + 2, A, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED
    assert st(A, A, A + 1, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED
    if "gemm" not in name:
        assert st(A, A, A, 9, 8, 256, None) == bad
    if name == "plm_quantize_gemv_q4K":   # f32 activations: 16-byte aligned
        assert st(A, A + 4, A, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED


def test_quantize_argument_checks():
    st = lambda *a: P.raw_status("plm_quantize_q8K", *a)  # noqa: E731
    bad = P.PLM_ERR_INVALID_ARG
    assert st(None, A, 1, 256, None) == bad
    assert st(A, None, 1, 256, None) == bad
    assert st(A, A, 0, 256, None) == bad
    assert st(A, A, 1, 255, None) == bad
    assert st(A + 4, A, 1, 256, None) == P.PLM_ERR_MISALIGNED
    assert st(A, A + 1, 1, 256, None) == P.PLM_ERR_MISALIGNED


def test_binding_raises_on_bad_arguments():
    with pytest.raises(q.PlmError, match="invalid argument"):
        q.plm_gemv_q4K(A, A, A, 9, 8, 256, stream=0)


def test_grouped_argument_checks():
    import ctypes
    lib = q.load()
    arr = (P._Problem * 2)()
    arr[0] = P._Problem(A, A, A, 8, 256)
    arr[1] = P._Problem(A, A, A, 8, 300)          # bad k in the second problem
    assert lib.plm_gemv_q4K_grouped(arr, 2, 1, None) == P.PLM_ERR_INVALID_ARG
    arr[1] = P._Problem(A + 8, A, A, 8, 256)      # misaligned w
    assert lib.plm_gemv_q6K_grouped(arr, 2, 1, None) == P.PLM_ERR_MISALIGNED
    assert lib.plm_gemv_q4K_grouped(arr, 0, 1, None) == P.PLM_ERR_INVALID_ARG
    assert lib.plm_gemv_q4K_grouped(arr, 1, 9, None) == P.PLM_ERR_INVALID_ARG
    assert lib.plm_gemv_q4K_grouped(None, 1, 1, None) == P.PLM_ERR_INVALID_ARG


def test_fused_grouped_argument_checks():
    lib = q.load()
    arr = (P._QProblem * 2)()
    arr[0] = P._QProblem(A, A, A, 8, 256)
    arr[1] = P._QProblem(A, A, A, 8, 300)          # bad k in the second problem
    assert lib.plm_quantize_gemv_q4K_grouped(arr, 2, 1, None) == P.PLM_ERR_INVALID_ARG
    arr[1] = P._QProblem(A, A + 8, A, 8, 256)      # x not 16-byte aligned
    assert lib.plm_quantize_gemv_q4K_grouped(arr, 2, 1, None) == P.PLM_ERR_MISALIGNED
    arr[1] = P._QProblem(A, A, A, 8, 256)
    assert lib.plm_quantize_gemv_q4K_grouped(arr, 0, 1, None) == P.PLM_ERR_INVALID_ARG
    assert lib.plm_quantize_gemv_q4K_grouped(arr, 2, 9, None) == P.PLM_ERR_INVALID_ARG
    assert lib.plm_quantize_gemv_q4K_grouped(None, 1, 1, None) == P.PLM_ERR_INVALID_ARG


def test_swiglu_argument_checks():
    lib = q.load()
    st = lambda *a: lib.plm_gemv_q4K_swiglu(*a)  # noqa: E731
    bad = P.PLM_ERR_INVALID_ARG
    assert st(None, A, A, A, 1, 8, 256, None) == bad
    assert st(A, None, A, A, 1, 8, 256, None) == bad
    assert st(A, A, None, A, 1, 8, 256, None) == bad
    assert st(A, A, A, None, 1, 8, 256, None) == bad
    assert st(A, A, A, A, 9, 8, 256, None) == bad
    assert st(A, A, A, A, 1, 8, 300, None) == bad
    assert st(A, A + 8, A, A, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED
    assert st(A + 8, A, A, A, 1, 8, 256, None) == P.PLM_ERR_MISALIGNED
    arr = (P._SProblem * 2)()
    arr[0] = P._SProblem(A, A, A, A, 8, 256)
    arr[1] = P._SProblem(A, A + 4, A, A, 8, 256)   # misaligned up matrix in the second pair
    assert lib.plm_gemv_q4K_swiglu_grouped(arr, 2, 1, None) == P.PLM_ERR_MISALIGNED
    assert lib.plm_gemv_q4K_swiglu_grouped(arr, 0, 1, None) == bad
    assert lib.plm_gemv_q4K_swiglu_grouped(None, 1, 1, None) == bad


def test_gemm_swiglu_argument_checks():
    lib = q.load()
    bad = P.PLM_ERR_INVALID_ARG
    for name in ("plm_gemm_q4K_swiglu", "plm_gemm_q4K_swiglu_ws"):
        ws = (A, 1 << 30) if name.endswith("_ws") else ()
        st = lambda *a: getattr(lib, name)(*(a[:7] + ws + a[7:]))  # noqa: E731
        assert st(None, A, A, A, 512, 8, 256, None) == bad
        assert st(A, None, A, A, 512, 8, 256, None) == bad
        assert st(A, A, None, A, 512, 8, 256, None) == bad
        assert st(A, A, A, None, 512, 8, 256, None) == bad
        assert st(A, A, A, A, 0, 8, 256, None) == bad
        assert st(A, A, A, A, 512, 0, 256, None) == bad
        assert st(A, A, A, A, 512, 8, 300, None) == bad
        assert st(A, A + 8, A, A, 512, 8, 256, None) == P.PLM_ERR_MISALIGNED
        assert st(A + 8, A, A, A, 512, 8, 256, None) == P.PLM_ERR_MISALIGNED
    # caller workspace: too small, or not 256-byte aligned
    need = q.plm_gemm_swiglu_workspace_size(512, 8, 256)
    assert need >= 512 * 8 * 4 + q.plm_gemm_workspace_size(4, 512, 256)
    assert q.plm_gemm_swiglu_workspace_size(8, 8, 256) == 0 and q.plm_gemm_swiglu_workspace_size(512, 8, 300) == 0
    assert lib.plm_gemm_q4K_swiglu_ws(A, A, A, A, 512, 8, 256, A, need - 1, None) == bad
    assert lib.plm_gemm_q4K_swiglu_ws(A, A, A, A, 512, 8, 256, None, need, None) == bad
    assert lib.plm_gemm_q4K_swiglu_ws(A, A, A, A, 512, 8, 256, A + 16, need, None) == P.PLM_ERR_MISALIGNED


def test_selftest_bounded_wait_rejects_bad_limits():
    # host-side checks only: nothing is launched for a rejected limit
    for rounds in (0, (1 << 16) + 1):
        assert P.raw_status("plm_selftest_bounded_wait", rounds, 0, None) == P.PLM_ERR_INVALID_ARG
