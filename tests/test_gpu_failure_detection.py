"""Failure detection on the GPU without a fault.

Every kernel that streams through asynchronous copies bounds its mbarrier
waits; a wait that runs out sets bit 0 of the library's device fault word
and the kernel returns instead of hanging.  plm_selftest_bounded_wait runs
that same bounded wait on a barrier nothing ever arrives at (no copy is
issued, nothing is left in flight), with a short limit, so the wait really
runs out.  The test checks that the word reports it, that clearing works,
that a wait that does complete leaves the word alone, and that the device is
still usable: a GEMV and a GEMM afterwards match the oracle.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import assert_close, gpu_matmul, oracle_ref

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    assert q.plm_device_fault() == 0                      # clean start (and cleared)
    q.plm_selftest_bounded_wait(64, complete=True)        # a wait that completes
    torch.cuda.synchronize()
    assert q.plm_device_fault(clear=False) == 0
    q.plm_selftest_bounded_wait(64, complete=False)       # nothing arrives: runs out
    torch.cuda.synchronize()
    assert q.plm_device_fault(clear=False) & 1 == 1
    assert q.plm_device_fault(clear=True) & 1 == 1         # read and clear
    assert q.plm_device_fault() == 0
    # the context is intact: normal calls still run and match the oracle
    for kind, m in (("gemv", 3), ("gemm", 40)):
        n, k = 70, 1024
        w = gen.q4K_blocks(50, 0, n, k)
        xq = oracle.quantize_q8K(gen.normal_f32(50, m, m, k))
        y = gpu_matmul(kind, "q4K", w, xq, m, n, k)
        ref, S = oracle_ref("q4K", w, xq, m, n, k)
        assert_close(y, ref, S)
    assert q.plm_device_fault() == 0

