"""Gate/up pair with the SwiGLU epilogue (plm_gemv_q4K_swiglu).

Two checks per case: (1) against silu applied in f64 to plm_gemv_q4K's own
outputs for each matrix -- the fused kernel forms the same f32 g and u, so
only its f32 epilogue (expf, add, divide, multiply) separates the two:
relative 1e-6; (2) against the oracle, h = silu(g) u in f64 on the oracle's
integer path, within the bound the GEMV tolerance implies:
|dh| <= 1.1 |u| dg + (|silu(g)| + 1.1 dg) du + 1e-6 |h|, with
dg = 1e-4 S_gate, du = 1e-4 S_up (|silu'| <= 1.1)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import TOL, dev, host

pytestmark = pytest.mark.gpu


def q8(x_np):
    m, k = x_np.shape
    xq = torch.empty(m * (k // 256) * 292, dtype=torch.uint8, device="cuda")
    q.plm_quantize_q8K(dev(x_np), xq, m, k)
    return xq


def gemv(w, xq, m, n, k):
    y = torch.full((m, n), float("nan"), device="cuda")
    q.plm_gemv_q4K(w, xq, y, m, n, k)
    return host(y)


def swiglu(wg, wu, xq, m, n, k):
    guard = 64
    hbuf = torch.full((m * n + guard,), float("nan"), device="cuda")
    hbuf[m * n:] = 12345.0
    q.plm_gemv_q4K_swiglu(wg, wu, xq, hbuf, m, n, k)
    out = host(hbuf)
    assert np.all(out[m * n:] == 12345.0), "write past the end of h"
    h = out[:m * n].reshape(m, n)
    assert not np.isnan(h).any(), "unwritten output elements"
    return h


def scaled_x(wg_np, seed, m, k):
    """Activations scaled so that the gate outputs land where silu bends (|g| ~ 2)."""
    x = gen.normal_f32(seed, 1, m, k)
    g = oracle.gemm_q4K_f64(wg_np, oracle.quantize_q8K(x), m, wg_np.shape[0], k)
    return (x * np.float32(2.0 / max(np.std(g), 1e-30))).astype(np.float32)


@pytest.mark.parametrize("n,k", [(64, 256), (3072, 1024), (257, 4096), (96, 12288)])
@pytest.mark.parametrize("m", [1, 3, 8])
def test_swiglu(n, k, m):
    wg_np = gen.q4K_blocks(60, n, n, k)
    wu_np = gen.q4K_blocks(61, n, n, k)
    x_np = scaled_x(wg_np, 60 + m, m, k)
    xq = q8(x_np)
    wg, wu = dev(wg_np), dev(wu_np)
    h = swiglu(wg, wu, xq, m, n, k).astype(np.float64)
    # (1) the epilogue on the GEMV's own g and u
    g, u = gemv(wg, xq, m, n, k), gemv(wu, xq, m, n, k)
    h_gemv = oracle.swiglu_f64(g, u)
    assert np.all(np.abs(h - h_gemv) <= 1e-6 * np.abs(h_gemv) + 1e-30)
    # (2) the oracle
    xq_ref = oracle.quantize_q8K(x_np)
    np.testing.assert_array_equal(host(xq).reshape(m, -1), xq_ref)
    g_ref = oracle.gemm_q4K_f64(wg_np, xq_ref, m, n, k)
    u_ref = oracle.gemm_q4K_f64(wu_np, xq_ref, m, n, k)
    h_ref = oracle.swiglu_f64(g_ref, u_ref)
    dg = TOL * oracle.absscale_q4K(wg_np, xq_ref, m, n, k)
    du = TOL * oracle.absscale_q4K(wu_np, xq_ref, m, n, k)
    bound = 1.1 * np.abs(u_ref) * dg + (np.abs(oracle.swiglu_f64(g_ref, np.ones_like(g_ref))) + 1.1 * dg) * du \
        + 1e-6 * np.abs(h_ref)
    assert np.all(np.abs(h - h_ref) <= bound)
    # the gate outputs do cover the bend of silu
    assert np.mean(np.abs(g_ref) < 4.0) > 0.5


def test_swiglu_grouped_equals_single():
    m = 2
    shapes = [(3072, 1024), (1024, 3072), (40, 256), (300, 9216)]
    probs, hs, singles = [], [], []
    for i, (n, k) in enumerate(shapes):
        wg_np, wu_np = gen.q4K_blocks(70 + i, 0, n, k), gen.q4K_blocks(70 + i, 1, n, k)
        xq = q8(scaled_x(wg_np, 70 + i, m, k))
        wg, wu = dev(wg_np), dev(wu_np)
        h = torch.full((m, n), float("nan"), device="cuda")
        probs.append((wg, wu, xq, h, n, k))
        hs.append(h)
        singles.append(swiglu(wg, wu, xq, m, n, k))
    q.plm_gemv_q4K_swiglu_grouped(probs, m)
    for h, s in zip(hs, singles):
        np.testing.assert_array_equal(host(h), s)
    assert q.plm_device_fault() == 0
