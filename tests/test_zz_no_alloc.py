"""The allocation-free GEMM entry points.

plm_gemm_q4K_noalloc runs the workspace form of the q4_K GEMM with its
workspace in a fixed device array inside the library; it must agree with
plm_gemm_q4K (which widens the activation codes inside the kernel, needs no
workspace and may split K over a cluster) -- bit for bit where neither
splits -- and match the oracle within the tolerance every GEMM test uses
(1e-4 of sum_k |w_hat * x_hat|).  No plain GEMM entry point may
draw on the device's stream-ordered pool.  This file is named so that pytest
collects it last.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from quant_packed_gemv_gb300 import plm as P
from tests.gpu_helpers import TOL, assert_close, dev, host, oracle_ref

pytestmark = pytest.mark.gpu


def _case(seed, m, n, k):
    w = gen.q4K_blocks(seed, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(seed, 5, m, k))
    return w, xq


def test_noalloc_matches_allocating_gemm_on_two_calls_in_a_row():
    cases = [(41, 300, 200, 2048), (42, 64, 130, 1024)]
    dev_in, outs = [], []
    for seed, m, n, k in cases:
        w, xq = _case(seed, m, n, k)
        dev_in.append((dev(w), dev(xq)))
        outs.append(torch.full((m, n), float("nan"), device="cuda"))
    # two calls in a row through the C ABI, the second reusing the array the
    # first wrote
    for (wd, xd), y, (_, m, n, k) in zip(dev_in, outs, cases):
        q.plm_gemm_q4K_noalloc(wd, xd, y, m, n, k)
    torch.cuda.synchronize()
    for (wd, xd), y, (seed, m, n, k) in zip(dev_in, outs, cases):
        y_alloc = torch.full((m, n), float("nan"), device="cuda")
        q.plm_gemm_q4K(wd, xd, y_alloc, m, n, k)
        got, want = host(y), host(y_alloc)
        w, xq = _case(seed, m, n, k)
        ref, S = oracle_ref("q4K", w, xq, m, n, k)
        assert not np.isnan(got).any()
        # plm_gemm_q4K may split K over a cluster where this entry does not: the tolerance
        assert np.all(np.abs(got.astype(np.float64) - want) <= TOL * S)
        assert_close(got, ref, S)
    assert q.plm_device_fault() == 0


def test_noalloc_small_m_runs_the_gemv():
    # m <= 8 needs no workspace: the call runs the decode GEMV, like plm_gemm_q4K
    for m in (1, 8):
        n, k = 96, 1024
        w, xq = _case(43, m, n, k)
        wd, xd = dev(w), dev(xq)
        y = torch.full((m, n), float("nan"), device="cuda")
        y_alloc = torch.full((m, n), float("nan"), device="cuda")
        q.plm_gemm_q4K_noalloc(wd, xd, y, m, n, k)
        q.plm_gemm_q4K(wd, xd, y_alloc, m, n, k)
        np.testing.assert_array_equal(host(y), host(y_alloc))


def test_noalloc_limit_edge():
    # workspace bytes = 2*m*k + 48*m*k/256, each part rounded up to 256: at
    # k = 256, m = 59918 needs 33,554,176 bytes (fits the 32 MiB array) and
    # m = 59919 needs 33,554,688 (one size up: rejected before any launch)
    k, n = 256, 64
    assert q.plm_gemm_workspace_size("q4K", 59918, k) <= P.PLM_NOALLOC_WORKSPACE_BYTES
    assert q.plm_gemm_workspace_size("q4K", 59919, k) > P.PLM_NOALLOC_WORKSPACE_BYTES
    m = 59918
    w, xq = _case(44, m, n, k)
    wd, xd = dev(w), dev(xq)
    y = torch.full((m, n), float("nan"), device="cuda")
    y_alloc = torch.full((m, n), float("nan"), device="cuda")
    q.plm_gemm_q4K_noalloc(wd, xd, y, m, n, k)
    q.plm_gemm_q4K(wd, xd, y_alloc, m, n, k)
    got, want = host(y), host(y_alloc)
    assert not np.isnan(got).any()
    rows = np.r_[0:64, m - 64:m]          # the first and last activation tiles against the oracle
    ref, S = oracle_ref("q4K", w, xq[rows], len(rows), n, k)
    assert_close(got[rows], ref, S)
    # one block of K: neither form splits, the same operands and sums, the same bits
    np.testing.assert_array_equal(got, want)
    st = P.raw_status("plm_gemm_q4K_noalloc", wd.data_ptr(), xd.data_ptr(), y.data_ptr(), m + 1, n, k, None)
    assert st == P.PLM_ERR_UNSUPPORTED


def test_noalloc_rejects_sizes_beyond_its_array():
    # about 2.19 * m * k bytes of workspace, above PLM_NOALLOC_WORKSPACE_BYTES (32 MiB)
    fake = 1 << 20   # never dereferenced: the call is rejected before any launch
    st = P.raw_status("plm_gemm_q4K_noalloc", fake, fake, fake, 2048, 256, 12288, None)
    assert st == P.PLM_ERR_UNSUPPORTED
    # argument checks come first: m = 0 is an invalid argument, not a size problem
    assert P.raw_status("plm_gemm_q4K_noalloc", fake, fake, fake, 0, 256, 256, None) == P.PLM_ERR_INVALID_ARG


def _pool_used_high():
    """High-water mark of the current device's default stream-ordered memory
    pool (the pool plm_gemm_q4K's cudaMallocAsync draws on), through the
    driver API; it is reset to the current use before returning."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    dev_h, pool = ctypes.c_int(0), ctypes.c_void_p(0)
    assert cu.cuDeviceGet(ctypes.byref(dev_h), torch.cuda.current_device()) == 0
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev_h) == 0
    used_high = 8                         # CU_MEMPOOL_ATTR_USED_MEM_HIGH
    val = ctypes.c_uint64(0)
    assert cu.cuMemPoolGetAttribute(pool, used_high, ctypes.byref(val)) == 0
    zero = ctypes.c_uint64(0)
    assert cu.cuMemPoolSetAttribute(pool, used_high, ctypes.byref(zero)) == 0
    return val.value


def _pool_alloc_free(nbytes):
    """Takes nbytes from the default pool and gives them back (driver API,
    legacy stream), to show that the high-water mark sees pool use."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    ptr = ctypes.c_uint64(0)
    assert cu.cuMemAllocAsync(ctypes.byref(ptr), ctypes.c_size_t(nbytes), None) == 0
    assert cu.cuMemFreeAsync(ptr, None) == 0
    assert cu.cuCtxSynchronize() == 0


def test_no_gemm_entry_draws_from_the_pool():
    m, n, k = 300, 200, 2048
    w, xq = _case(45, m, n, k)
    wd, xd = dev(w), dev(xq)
    w5 = dev(gen.q5K_blocks(45, 0, n, k))
    w6 = dev(gen.q6K_blocks(45, 0, n, k))
    wu = dev(gen.q4K_blocks(46, 0, n, k))
    y = torch.full((m, n), float("nan"), device="cuda")
    torch.cuda.synchronize()
    _pool_used_high()                     # reset the high-water mark
    for _ in range(2):
        q.plm_gemm_q4K_noalloc(wd, xd, y, m, n, k)
        q.plm_gemm_q4K(wd, xd, y, m, n, k)
        q.plm_gemm_q5K(w5, xd, y, m, n, k)
        q.plm_gemm_q6K(w6, xd, y, m, n, k)
        q.plm_gemm_q4K_swiglu(wd, wu, xd, y, m, n, k)
    torch.cuda.synchronize()
    assert _pool_used_high() == 0
    assert q.plm_device_fault() == 0
    # the measurement does see memory taken from the pool
    _pool_alloc_free(1 << 20)
    assert _pool_used_high() >= 1 << 20
