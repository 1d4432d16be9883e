"""GPU parity of the row-interleaved q4_K and q6_K layouts (x16) and their
tensor-core decode GEMV, through the C ABI.

The repack is bit-exact against the test-side packer written from the layout
definition; the GEMV on the repacked weights is compared with the oracle on
the original q4_K blocks, element by element at 1e-4 of sum_k |w_hat * x_hat|
(every m = 1..8, ragged row counts, block counts that give every team shape:
nb odd, 4, 12, 16, 48), at the extremes of the codes, and at the Qwen3-8B
shapes on sampled rows.  Activation row i gives the same bits at every m."""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import assert_close, dev, host, oracle_ref
from tests.packers import pack_q4K, pack_q4K_x16, pack_q6K, pack_q6K_x16

pytestmark = pytest.mark.gpu


def repack(w_np, n, k, fmt="q4K"):
    wx = torch.full((getattr(q, "plm_%s_x16_size" % fmt)(n, k),), 0xA5, dtype=torch.uint8, device="cuda")
    getattr(q, "plm_%s_to_x16" % fmt)(dev(w_np), wx, n, k)
    return wx


def gemv_x16(wx, xq_np, m, n, k, fmt="q4K"):
    guard = 64
    ybuf = torch.full((m * n + guard,), float("nan"), dtype=torch.float32, device="cuda")
    ybuf[m * n:] = 12345.0
    getattr(q, "plm_gemv_%s_x16" % fmt)(wx, dev(xq_np), ybuf, m, n, k)
    out = host(ybuf)
    assert np.all(out[m * n:] == 12345.0), "write past the end of y"
    y = out[:m * n].reshape(m, n)
    assert not np.isnan(y).any(), "unwritten output elements"
    return y


@pytest.mark.parametrize("n,k", [(1, 256), (16, 512), (37, 1024), (300, 2816), (130, 12288)])
def test_repack_bit_exact(n, k):
    w = gen.q4K_blocks(80, 0, n, k)
    np.testing.assert_array_equal(host(repack(w, n, k)), pack_q4K_x16(w, n, k))


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n,k", [(1, 256), (37, 1024), (100, 1280), (64, 3072), (200, 4096), (33, 12288)])
def test_gemv_x16_matches_oracle(m, n, k):
    w = gen.q4K_blocks(81, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(81, 300 + m, m, k))
    y = gemv_x16(repack(w, n, k), xq, m, n, k)
    ref, S = oracle_ref("q4K", w, xq, m, n, k)
    assert_close(y, ref, S)


def test_gemv_x16_row_result_independent_of_m():
    n, k = 300, 4096
    w = gen.q4K_blocks(82, 0, n, k)
    wx = repack(w, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(82, 1, 8, k))
    y8 = gemv_x16(wx, xq, 8, n, k)
    for i in range(8):
        np.testing.assert_array_equal(gemv_x16(wx, xq[i:i + 1], 1, n, k)[0], y8[i])
    np.testing.assert_array_equal(gemv_x16(wx, xq[2:5], 3, n, k), y8[2:5])


def test_gemv_x16_adversarial_extremes():
    k, n, m = 2048, 40, 8
    blocks = [pack_q4K(2e-3, 2e-3, [63] * 8, [63] * 8, np.full(256, 15)),
              pack_q4K(2e-3, 2e-3, [63] * 8, [63] * 8, np.zeros(256)),
              pack_q4K(1e-4, 2e-3, [63, 0] * 4, [0, 63] * 4, 15 * np.tile([0, 1], 128))]
    w = np.stack([np.concatenate([blocks[(r + b) % 3] for b in range(k // 256)]) for r in range(n)])
    x = np.full((m, k), -1.0, dtype=np.float32)
    x[1] = 1.0
    x[2, ::2] = 1.0
    x[3:] = gen.normal_f32(83, 0, m - 3, k)
    xq = oracle.quantize_q8K(x)
    y = gemv_x16(repack(w, n, k), xq, m, n, k)
    ref, S = oracle_ref("q4K", w, xq, m, n, k)
    assert_close(y, ref, S)


@pytest.mark.parametrize("n,k", [(12288, 4096), (4096, 12288)])
@pytest.mark.parametrize("m", [1, 8])
def test_gemv_x16_qwen3_8b_shapes(n, k, m):
    # full-size weights (seed 4, as the bench), oracle on sampled rows
    w = gen.q4K_blocks(4, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(4, 9, m, k))
    y = gemv_x16(repack(w, n, k), xq, m, n, k)
    rng = np.random.default_rng(n + m)
    rows = np.unique(np.concatenate([rng.choice(n, 40, replace=False), np.arange(16), np.arange(n - 16, n)]))
    nb = k // 256
    ws = w.reshape(n, nb * 144)[rows]
    ref, S = oracle_ref("q4K", ws, xq, m, len(rows), k)
    assert_close(y[:, rows], ref, S)
    assert q.plm_device_fault() == 0


# ---------------------------------------------------------------- q6_K

@pytest.mark.parametrize("n,k", [(1, 256), (16, 512), (37, 1024), (300, 2816), (130, 12288)])
def test_q6K_repack_bit_exact(n, k):
    w = gen.q6K_blocks(84, 0, n, k)
    np.testing.assert_array_equal(host(repack(w, n, k, "q6K")), pack_q6K_x16(w, n, k))


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n,k", [(1, 256), (37, 1024), (100, 1280), (64, 3072), (200, 4096), (33, 12288)])
def test_gemv_q6K_x16_matches_oracle(m, n, k):
    w = gen.q6K_blocks(85, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(85, 300 + m, m, k))
    y = gemv_x16(repack(w, n, k, "q6K"), xq, m, n, k, "q6K")
    ref, S = oracle_ref("q6K", w, xq, m, n, k)
    assert_close(y, ref, S)


def test_gemv_q6K_x16_row_result_independent_of_m():
    n, k = 300, 4096
    w = gen.q6K_blocks(86, 0, n, k)
    wx = repack(w, n, k, "q6K")
    xq = oracle.quantize_q8K(gen.normal_f32(86, 1, 8, k))
    y8 = gemv_x16(wx, xq, 8, n, k, "q6K")
    for i in range(8):
        np.testing.assert_array_equal(gemv_x16(wx, xq[i:i + 1], 1, n, k, "q6K")[0], y8[i])


def test_gemv_q6K_x16_adversarial_extremes():
    # every int8 scale extreme (the largest |sc * (q6 - 32)| is 4096, not exact
    # in f16: the kernel scales the exact group dot in f32 instead)
    k, n, m = 2048, 40, 8
    alt = np.tile([0, 63], 128)
    blocks = [pack_q6K(2e-3, [-128] * 16, np.zeros(256)), pack_q6K(2e-3, [127] * 16, np.full(256, 63)),
              pack_q6K(2e-3, [-64] * 16, np.full(256, 63)), pack_q6K(2e-3, [-128, 127, -1, 65] * 4, alt),
              pack_q6K(2e-3, [5] * 16, np.full(256, 32))]
    w = np.stack([np.concatenate([blocks[(r + b) % 5] for b in range(k // 256)]) for r in range(n)])
    x = np.full((m, k), -1.0, dtype=np.float32)
    x[1] = 1.0
    x[2, ::2] = 1.0
    x[3:] = gen.normal_f32(87, 0, m - 3, k)
    xq = oracle.quantize_q8K(x)
    y = gemv_x16(repack(w, n, k, "q6K"), xq, m, n, k, "q6K")
    ref, S = oracle_ref("q6K", w, xq, m, n, k)
    assert_close(y, ref, S)


@pytest.mark.parametrize("k", [2048, 4096])
@pytest.mark.parametrize("m", [1, 8])
def test_gemv_q6K_x16_output_heads(k, m):
    # the q6_K heads 151936 x 2048 (seed 3) and x 4096 (seed 4), oracle on sampled rows
    n = 151936
    w = gen.q6K_blocks(3 if k == 2048 else 4, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(4, 9, m, k))
    y = gemv_x16(repack(w, n, k, "q6K"), xq, m, n, k, "q6K")
    rng = np.random.default_rng(k + m)
    rows = np.unique(np.concatenate([rng.choice(n, 40, replace=False), np.arange(16), np.arange(n - 16, n)]))
    ws = w.reshape(n, (k // 256) * 210)[rows]
    ref, S = oracle_ref("q6K", ws, xq, m, len(rows), k)
    assert_close(y[:, rows], ref, S)
    assert q.plm_device_fault() == 0
