"""The allocation-free q4_K GEMM (plm_gemm_q4K_noalloc).

It serves callers that must not allocate device memory while running: its
workspace is a fixed device array inside the library rather than memory
taken from the stream-ordered pool.  Its results must agree with
plm_gemm_q4K, which allocates its workspace, within the tolerance every GEMM
test uses (1e-4 of sum_k |w_hat * x_hat|).  This file is named so that
pytest collects it last.
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
        assert np.all(np.abs(got.astype(np.float64) - want) <= TOL * S)
        assert_close(got, ref, S)
    assert q.plm_device_fault() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    # about 2.19 * m * k bytes of workspace, above PLM_NOALLOC_WORKSPACE_BYTES (32 MiB)
    fake = 1 << 20   # never dereferenced: the call is rejected before any launch
    st = P.raw_status("plm_gemm_q4K_noalloc", fake, fake, fake, 2048, 256, 12288, None)
    assert st == P.PLM_ERR_UNSUPPORTED
    # small m needs no workspace at all
    assert P.raw_status("plm_gemm_q4K_noalloc", fake, fake, fake, 0, 256, 256, None) == P.PLM_ERR_INVALID_ARG
