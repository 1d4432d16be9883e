"""The device probe behind the GEMM's context figures: the tcgen05 MMA the
GEMM issues (kind::f16, 128 x 128 x 16, A from tensor memory) streams at the
dense rate when its issuing thread does nothing else, and an mbarrier wait
after each commit costs the tensor pipe.  Bounds are loose: cycles are SM
cycles (clock-independent), the rate only has to be of the right order."""
import pytest

import quant_packed_gemv_gb300 as q

pytestmark = pytest.mark.gpu


def test_tcgen05_rate_probe():
    cyc, cyc_wait, tflops = q.plm_probe_tcgen05_rate()
    # 2 * 128 * 128 * 16 flops at the nominal 8192 dense f16 flops per SM cycle: 64 cycles
    assert 40.0 <= cyc <= 100.0, cyc
    assert cyc_wait > cyc, (cyc, cyc_wait)
    assert tflops > 200.0, tflops
    assert q.plm_device_fault() == 0
