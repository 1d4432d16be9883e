"""Fused q8_K producer + q4_K GEMV (plm_quantize_gemv_q4K): the kernel
quantizes f32 activations itself.  It must give y bit for bit equal to the
two-step path (plm_quantize_q8K, whose bytes are pinned to the oracle, then
plm_gemv_q4K), and y within the tolerance of the oracle's f64 result on the
oracle's own q8_K codes."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import TOL, dev, host

pytestmark = pytest.mark.gpu


def two_step(w, x, m, n, k):
    xq = torch.empty(m * (k // 256) * 292, dtype=torch.uint8, device="cuda")
    q.plm_quantize_q8K(x, xq, m, k)
    y = torch.full((m, n), float("nan"), device="cuda")
    q.plm_gemv_q4K(w, xq, y, m, n, k)
    return host(y)


def fused(w, x, m, n, k):
    guard = 64
    ybuf = torch.full((m * n + guard,), float("nan"), device="cuda")
    ybuf[m * n:] = 12345.0
    q.plm_quantize_gemv_q4K(w, x, ybuf, m, n, k)
    out = host(ybuf)
    assert np.all(out[m * n:] == 12345.0), "write past the end of y"
    y = out[:m * n].reshape(m, n)
    assert not np.isnan(y).any(), "unwritten output elements"
    return y


@pytest.mark.parametrize("n,k", [(64, 256), (257, 1024), (1024, 3072), (300, 4096), (96, 12288)])
@pytest.mark.parametrize("m", [1, 2, 5, 8])
def test_fused_equals_two_step_and_oracle(n, k, m):
    w_np = gen.q4K_blocks(31, n + k, n, k)
    x_np = gen.normal_f32(31, 500 + m, m, k)
    w, x = dev(w_np), dev(x_np)
    yf = fused(w, x, m, n, k)
    np.testing.assert_array_equal(yf, two_step(w, x, m, n, k))
    xq = oracle.quantize_q8K(x_np)
    ref = oracle.gemm_q4K_f64(w_np, xq, m, n, k)
    S = oracle.absscale_q4K(w_np, xq, m, n, k)
    assert np.all(np.abs(yf.astype(np.float64) - ref) <= TOL * S)


def test_fused_adversarial_activations():
    """All-zero chunks, amax ties of both signs, exact .5 products and huge or
    tiny magnitudes go through the in-kernel quantizer unchanged."""
    n, k, m = 128, 2048, 3
    x_np = gen.normal_f32(7, 1, m, k)
    x_np[0, :256] = 0.0                       # all-zero chunk
    x_np[1, 256:512] = 0.0
    x_np[1, 300] = -3.0
    x_np[1, 301] = 3.0                        # tie on |max|, negative first
    x_np[2, 512:768] = np.linspace(-1.0, 1.0, 256, dtype=np.float32)
    x_np[2, 1024:1280] *= 1e30
    x_np[2, 1280:1536] *= 1e-30
    w_np = gen.q4K_blocks(7, 2, n, k)
    w, x = dev(w_np), dev(x_np)
    yf = fused(w, x, m, n, k)
    np.testing.assert_array_equal(yf, two_step(w, x, m, n, k))


def test_fused_grouped_equals_single():
    rng = np.random.default_rng(3)
    shapes = [(2048, 1024), (1024, 1024), (1024, 2048), (3072, 1024), (1024, 3072), (40, 256), (512, 8192)]
    m = 2
    ws, xs, ys, probs, singles = [], [], [], [], []
    for i, (n, k) in enumerate(shapes):
        w = dev(gen.q4K_blocks(40 + i, 0, n, k))
        x = dev(gen.normal_f32(40 + i, 1, m, k) * np.float32(rng.uniform(0.1, 10)))
        y = torch.full((m, n), float("nan"), device="cuda")
        ws.append(w), xs.append(x), ys.append(y)
        probs.append((w, x, y, n, k))
        singles.append(fused(w, x, m, n, k))
    q.plm_quantize_gemv_q4K_grouped(probs, m)
    for y, s in zip(ys, singles):
        np.testing.assert_array_equal(host(y), s)
    assert q.plm_device_fault() == 0


def test_fused_decode_set_grouped():
    """The 196-matrix Qwen3-0.6B decode set through one fused grouped launch:
    bit-equal to the two-step grouped path."""
    import bench
    mats, host_w, xs = bench.host_inputs()
    w_dev = torch.from_numpy(host_w).cuda()
    fprobs, gprobs, yf, yg = [], [], [], []
    for idx, (_, _, n, k, off) in enumerate(mats):
        x = dev(xs[idx])
        xq = torch.empty(k // 256 * 292, dtype=torch.uint8, device="cuda")
        q.plm_quantize_q8K(x, xq, 1, k)
        a = torch.full((n,), float("nan"), device="cuda")
        b = torch.full((n,), float("nan"), device="cuda")
        fprobs.append((w_dev.data_ptr() + off, x, a, n, k))
        gprobs.append((w_dev.data_ptr() + off, xq, b, n, k))
        yf.append(a), yg.append(b)
        xs[idx] = x            # keep the device copies alive
    q.plm_quantize_gemv_q4K_grouped(fprobs, 1)
    q.plm_gemv_q4K_grouped(gprobs, 1)
    for a, b in zip(yf, yg):
        np.testing.assert_array_equal(host(a), host(b))


@pytest.mark.parametrize("m", [1, 4])
def test_fused_reads_and_writes_pinned_host_memory(m):
    # x and y in pinned host memory, which the GPU reaches directly: the same
    # bits as with device buffers (the end-to-end zero-copy measurement)
    n, k = 300, 2048
    w = dev(gen.q4K_blocks(43, 0, n, k))
    x_np = gen.normal_f32(43, 1, m, k)
    x_host = torch.from_numpy(x_np).pin_memory()
    y_host = torch.full((m, n), float("nan")).pin_memory()
    q.plm_quantize_gemv_q4K_grouped([(w, x_host.data_ptr(), y_host.data_ptr(), n, k)], m)
    torch.cuda.synchronize()
    want = fused(w, torch.from_numpy(x_np).cuda(), m, n, k)
    np.testing.assert_array_equal(y_host.numpy(), want)
