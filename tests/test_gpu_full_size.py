"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times.  Where the oracle would take minutes, it is computed on sampled
output rows (weight rows are independent, so a slice of W gives exactly
those outputs); the q8_K bytes are always compared in full.

Workloads (seeded synthetic, the shapes of the Qwen3 models the PocketLLM
pages run):
  q4_K 1024x1024 at m=1 (seed 0); the Qwen3-0.6B decode set of 196 matrices
  through the grouped GEMV (seed 1); m=512 prefill GEMMs 1024x1024,
  6144x2048, 2048x6144 (seed 2); the q6_K head 151936x2048 at m = 1, 8, 512
  (seed 3); the Qwen3-8B shapes 12288x4096, 4096x12288 and the q6_K head
  151936x4096 over m = 1..2048 (seed 4).
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q
from tests.gpu_helpers import TOL, dev, host

pytestmark = pytest.mark.gpu

BYTES = {"q4K": 144, "q6K": 210}


def weights(fmt, seed, n, k):
    return gen.q4K_blocks(seed, 0, n, k) if fmt == "q4K" else gen.q6K_blocks(seed, 0, n, k)


def sample_rows(n, count=48, seed=0):
    rng = np.random.default_rng(seed + n)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update(range(max(0, n - 8), n))      # the last rows (last tile)
    rows.update(range(min(8, n)))
    return np.array(sorted(rows))


def run_gpu(fmt, w_dev, x_np, n, k):
    """Quantize x on the GPU (checked bit-exact) and run the entry point the
    bench times for this m: GEMV for m <= 8, GEMM (workspace form) above."""
    m = x_np.shape[0]
    xq = torch.empty(m * (k // 256) * 292, dtype=torch.uint8, device="cuda")
    q.plm_quantize_q8K(dev(x_np), xq, m, k)
    xq_ref = oracle.quantize_q8K(x_np)
    np.testing.assert_array_equal(host(xq).reshape(m, -1), xq_ref)
    y = torch.full((m, n), float("nan"), device="cuda")
    if m <= 8:
        getattr(q, "plm_gemv_%s" % fmt)(w_dev, xq, y, m, n, k)
    else:
        need = q.plm_gemm_workspace_size(fmt, m, k)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        getattr(q, "plm_gemm_%s_ws" % fmt)(w_dev, xq, y, m, n, k, ws, need)
    out = host(y)
    assert not np.isnan(out).any()
    return out, xq_ref


def check_rows(fmt, w_np, xq_ref, y, rows, k):
    m = y.shape[0]
    wr = np.ascontiguousarray(w_np[rows])
    ref = getattr(oracle, "gemm_%s_f64" % fmt)(wr, xq_ref, m, len(rows), k)
    S = getattr(oracle, "absscale_%s" % fmt)(wr, xq_ref, m, len(rows), k)
    err = np.abs(y[:, rows].astype(np.float64) - ref)
    assert np.all(err <= TOL * S), float((err / S).max())


def test_config0_q4K_1024x1024_m1_full():
    n = k = 1024
    w = weights("q4K", 0, n, k)
    x = gen.normal_f32(0, 1, 1, k)
    y, xq = run_gpu("q4K", dev(w), x, n, k)
    check_rows("q4K", w, xq, y, np.arange(n), k)


def test_config1_decode_set_grouped():
    import bench
    mats, host_w, xs = bench.host_inputs()
    w_dev = torch.from_numpy(host_w).cuda()
    xq_list, probs, ys = [], [], []
    for idx, (_, _, n, k, off) in enumerate(mats):
        xq = torch.empty(k // 256 * 292, dtype=torch.uint8, device="cuda")
        q.plm_quantize_q8K(dev(xs[idx]), xq, 1, k)
        y = torch.full((n,), float("nan"), device="cuda")
        probs.append((w_dev.data_ptr() + off, xq, y, n, k))
        xq_list.append(xq)
        ys.append(y)
    q.plm_gemv_q4K_grouped(probs, 1)
    torch.cuda.synchronize()
    for idx, (layer, _, n, k, off) in enumerate(mats):
        xq_ref = oracle.quantize_q8K(xs[idx])
        np.testing.assert_array_equal(host(xq_list[idx]), xq_ref.ravel())
        w = host_w[off:off + n * (k // 256) * 144].reshape(n, -1)
        rows = np.arange(n) if layer in (0, 27) else sample_rows(n, 12, idx)
        check_rows("q4K", w, xq_ref, host(ys[idx]).reshape(1, n), rows, k)


@pytest.mark.parametrize("n,k", [(1024, 1024), (6144, 2048), (2048, 6144)])
def test_config2_prefill_gemm_m512(n, k):
    w = weights("q4K", 2, n, k)
    x = gen.normal_f32(2, 7, 512, k)
    y, xq = run_gpu("q4K", dev(w), x, n, k)
    rows = np.arange(n) if n * k <= 1 << 20 else sample_rows(n, 48)
    check_rows("q4K", w, xq, y, rows, k)


@pytest.fixture(scope="module")
def head2048():
    w = weights("q6K", 3, 151936, 2048)
    return w, dev(w)


@pytest.mark.parametrize("m", [1, 8, 512])
def test_config3_q6K_head(head2048, m):
    w, w_dev = head2048
    n, k = 151936, 2048
    x = gen.normal_f32(3, 11 + m, m, k)
    y, xq = run_gpu("q6K", w_dev, x, n, k)
    check_rows("q6K", w, xq, y, sample_rows(n, 64), k)


@pytest.mark.parametrize("fmt,n,k", [("q4K", 12288, 4096), ("q4K", 4096, 12288), ("q6K", 151936, 4096)])
def test_config4_qwen3_8b_sweep(fmt, n, k):
    w = weights(fmt, 4, n, k)
    w_dev = dev(w)
    for m in (1, 2, 4, 8, 64, 512, 2048):
        # the q6_K head at m = 2048: 1.27e12 MACs on the GPU, a 1.2 GB result; the oracle
        # takes the sampled rows only
        x = gen.normal_f32(4, 100 + m, m, k)
        y, xq = run_gpu(fmt, w_dev, x, n, k)
        check_rows(fmt, w, xq, y, sample_rows(n, 16 if m >= 512 else 32, m), k)
    assert q.plm_device_fault() == 0
