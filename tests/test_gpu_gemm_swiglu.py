"""Prefill gate/up pair with the SwiGLU epilogue (plm_gemm_q4K_swiglu).

As for the decode pair: (1) against silu applied in f64 to the plain q4_K
GEMM's own outputs for each matrix (the pair computes the same f32 g and u;
m <= 8: the GEMV's) -- relative 1e-6; (2) against the oracle, h = silu(g) u
in f64 on the oracle's integer path, within the bound the GEMM tolerance
implies: |dh| <= 1.1 |u| dg + (|silu(g)| + 1.1 dg) du + 1e-6 |h|, with
dg = 1e-4 S_gate, du = 1e-4 S_up (|silu'| <= 1.1).  The caller-workspace form
gives the same bits when it splits K as the plain form does."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import TOL, dev, host

pytestmark = pytest.mark.gpu


def scaled_x(wg_np, seed, m, k):
    """Activations scaled so that the gate outputs land where silu bends (|g| ~ 2)."""
    x = gen.normal_f32(seed, 1, m, k)
    g = oracle.gemm_q4K_f64(wg_np, oracle.quantize_q8K(x), m, wg_np.shape[0], k)
    return (x * np.float32(2.0 / max(np.std(g), 1e-30))).astype(np.float32)


def poisoned(m, n):
    guard = 64
    buf = torch.full((m * n + guard,), float("nan"), device="cuda")
    buf[m * n:] = 12345.0
    return buf


def unpoison(buf, m, n):
    out = host(buf)
    assert np.all(out[m * n:] == 12345.0), "write past the end of h"
    h = out[:m * n].reshape(m, n)
    assert not np.isnan(h).any(), "unwritten output elements"
    return h


def single(w, xq, m, n, k):
    """The matrix alone, in the same f32 order as the plain pair: the plain
    GEMM (the same K split), or the GEMV for m <= 8."""
    y = torch.full((m, n), float("nan"), device="cuda")
    if m <= 8:
        q.plm_gemv_q4K(w, xq, y, m, n, k)
    else:
        q.plm_gemm_q4K(w, xq, y, m, n, k)
    return host(y).astype(np.float64)


@pytest.mark.parametrize("m,n,k", [(512, 256, 1024), (300, 200, 2048), (9, 128, 256), (4, 100, 512),
                                   (1000, 256, 2048), (130, 1024, 3072), (640, 4096, 2048)])
def test_gemm_swiglu(m, n, k):
    # (640, 4096, 2048): 160 output tiles on 152 SMs, the last weight-tile rows
    # as a second launch with K split over clusters
    wg_np = gen.q4K_blocks(70, n, n, k)
    wu_np = gen.q4K_blocks(71, n, n, k)
    x_np = scaled_x(wg_np, 70 + m, m, k)
    xq_ref = oracle.quantize_q8K(x_np)
    xq = dev(xq_ref)
    wg, wu = dev(wg_np), dev(wu_np)
    hb = poisoned(m, n)
    q.plm_gemm_q4K_swiglu(wg, wu, xq, hb, m, n, k)
    h = unpoison(hb, m, n).astype(np.float64)
    # (1) the epilogue on the single-matrix outputs
    h_own = oracle.swiglu_f64(single(wg, xq, m, n, k), single(wu, xq, m, n, k))
    assert np.all(np.abs(h - h_own) <= 1e-6 * np.abs(h_own) + 1e-30)
    # (2) the oracle
    g_ref = oracle.gemm_q4K_f64(wg_np, xq_ref, m, n, k)
    u_ref = oracle.gemm_q4K_f64(wu_np, xq_ref, m, n, k)
    h_ref = oracle.swiglu_f64(g_ref, u_ref)
    dg = TOL * oracle.absscale_q4K(wg_np, xq_ref, m, n, k)
    du = TOL * oracle.absscale_q4K(wu_np, xq_ref, m, n, k)
    bound = 1.1 * np.abs(u_ref) * dg + (np.abs(oracle.swiglu_f64(g_ref, np.ones_like(g_ref))) + 1.1 * dg) * du \
        + 1e-6 * np.abs(h_ref)
    assert np.all(np.abs(h - h_ref) <= bound)
    assert np.mean(np.abs(g_ref) < 4.0) > 0.5   # the gate outputs do cover the bend of silu
    # caller workspace: with the split-K size (K split as the plain form splits
    # it over a cluster) the same bits -- the plain form combines in the up
    # GEMM's epilogue, the _ws form in a separate pass; unsplit within the bound
    split = q.plm_gemm_swiglu_workspace_size(m, n, k)
    unsplit = 0 if split == 0 else -(-m * n * 4 // 256) * 256 + q.plm_gemm_workspace_size("q4K", m, k)
    for need in sorted({unsplit, split}):
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        hb2 = poisoned(m, n)
        q.plm_gemm_q4K_swiglu_ws(wg, wu, xq, hb2, m, n, k, ws if need else None, need)
        h2 = unpoison(hb2, m, n)
        if need == split:
            assert np.array_equal(h2, h.astype(np.float32))
        assert np.all(np.abs(h2.astype(np.float64) - h_ref) <= bound)
    assert q.plm_device_fault() == 0
