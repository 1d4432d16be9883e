"""GPU parity: the CUDA library, called through its C ABI, against the oracle
on the same seeded inputs.  Integer results (q8_K bytes, sub-block dots) must
be bit-exact; f32 outputs must be within 1e-4 of sum_k |w_hat * x_hat|."""
import numpy as np
import pytest

import gen
import oracle
from tests.gpu_helpers import (assert_close, gpu_matmul, gpu_quantize, gpu_subdots, host,
                               make_weights, oracle_ref)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------- q8_K bytes

@pytest.mark.parametrize("seed,m,k", [(0, 1, 1024), (1, 7, 2048), (2, 512, 1024), (3, 3, 256),
                                      (4, 2, 12288)])
def test_quantize_bit_exact(seed, m, k):
    x = gen.normal_f32(seed, 100, m, k)
    x[0, :256:5] = 0.0
    x[-1, 256 % k:512 % k or k] = 0.0         # an all-zero chunk (or a zero run)
    mx = np.abs(x[0, :256]).max()
    x[0, 3], x[0, 7] = -mx, mx                # a magnitude tie, opposite signs
    np.testing.assert_array_equal(host(gpu_quantize(x)), oracle.quantize_q8K(x))


def test_quantize_scaled_and_tiny_values():
    x = gen.normal_f32(5, 1, 4, 1024)
    x[1] *= 1e-30
    x[2] *= 3e30
    x[3] = np.round(x[3] * 4) / 4            # many exact ties after scaling
    np.testing.assert_array_equal(host(gpu_quantize(x)), oracle.quantize_q8K(x))


# ------------------------------------------------------ integer sub-dots

@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
@pytest.mark.parametrize("m,n,k", [(1, 1, 256), (1, 33, 1024), (3, 17, 1280), (8, 40, 2048),
                                   (5, 9, 2816)])
def test_subdots_bit_exact(fmt, m, n, k):
    w = make_weights(fmt, 7, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(7, 200, m, k))
    got = gpu_subdots(fmt, w, xq, m, n, k)
    want = getattr(oracle, "subdots_%s" % fmt)(w, xq, m, n, k)
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------- GEMV

@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n,k", [(1, 256), (37, 1024), (100, 1280), (64, 3072), (37, 2048)])
def test_gemv_matches_oracle(fmt, m, n, k):
    # k = 2048 (8 blocks a row): q2_K, q3_K and q6_K on the one-lane-per-block
    # kernel, 37 rows leaving a partial stage; the other k: q3_K and q6_K on
    # the four-lanes-per-block kernel
    w = make_weights(fmt, 11, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(11, 300 + m, m, k))
    y = gpu_matmul("gemv", fmt, w, xq, m, n, k)
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    assert_close(y, ref, S)


@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
def test_gemv_row_result_independent_of_m(fmt):
    # the pages' tiled kernels are bit-identical to the single-row kernel;
    # here activation row i must give the same bits at every m.  For q3_K at
    # k = 2048 this also holds the one-lane kernel's two decodes to each other:
    # codes kept in place for m <= 3, shifted down for m > 3
    n, k = 300, 2048
    w = make_weights(fmt, 12, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(12, 1, 8, k))
    y8 = gpu_matmul("gemv", fmt, w, xq, 8, n, k)
    for i in range(8):
        y1 = gpu_matmul("gemv", fmt, w, xq[i:i + 1], 1, n, k)
        np.testing.assert_array_equal(y1[0], y8[i])


@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K", "q6K+"])
@pytest.mark.parametrize("k", [1024, 2048])
def test_gemv_adversarial_extremes(fmt, k):
    # all codes at the extremes: largest integer sums the formats allow, on
    # both decode kernels of q3_K and q6_K (k = 2048: one lane per block)
    from tests.packers import pack_q2K, pack_q3K, pack_q4K, pack_q5K, pack_q6K
    n, m = 8, 2
    if fmt == "q2K":
        blk = pack_q2K(2e-3, 2e-3, [15] * 16, [15] * 16, np.full(256, 3))
    elif fmt == "q3K":
        blk = pack_q3K(2e-3, [0] * 16, np.full(256, -4))      # scale -32, code -4
    elif fmt == "q4K":
        blk = pack_q4K(2e-3, 2e-3, [63] * 8, [63] * 8, np.full(256, 15))
    elif fmt == "q5K":
        blk = pack_q5K(2e-3, 2e-3, [63] * 8, [63] * 8, np.full(256, 31))
    elif fmt == "q6K":
        blk = pack_q6K(2e-3, [-64] * 16, np.zeros(256, dtype=np.int64))   # scale -64, q6 - 32 = -32
    else:
        blk = pack_q6K(2e-3, [127] * 16, np.full(256, 63))                 # scale 127, q6 - 32 = 31
        fmt = "q6K"
    w = np.tile(blk, n * k // 256).reshape(n, -1)
    x = np.full((m, k), -1.0, dtype=np.float32)
    x[1, ::2] = 1.0
    xq = oracle.quantize_q8K(x)
    y = gpu_matmul("gemv", fmt, w, xq, m, n, k)
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    assert_close(y, ref, S)


# --------------------------------------------------------------- GEMM

@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
@pytest.mark.parametrize("m,n,k", [(9, 50, 1024), (17, 33, 256), (64, 128, 2048), (130, 70, 512),
                                   (128, 128, 256), (200, 300, 1536), (512, 1024, 1024), (257, 129, 4096)])
def test_gemm_matches_oracle(fmt, m, n, k):
    w = make_weights(fmt, 13, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(13, 400, m, k))
    y = gpu_matmul("gemm", fmt, w, xq, m, n, k)
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    assert_close(y, ref, S)


@pytest.mark.parametrize("fmt", ["q4K", "q5K", "q6K"])
@pytest.mark.parametrize("shift", [4, 8, 12])
def test_gemm_xq_4_byte_aligned(fmt, shift):
    """xq needs only 4-byte alignment.  Off a 16-byte boundary the plain GEMM
    stages the activation codes with one bulk copy per row (each from the
    16-byte boundary at or below the row's codes) instead of one TMA box per
    block: the same bits as with an aligned xq."""
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import dev
    m, n, k = 140, 136, 2048
    w = make_weights(fmt, 15, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(15, 3, m, k))
    wd = dev(w)
    buf = torch.zeros(xq.nbytes + 64, dtype=torch.uint8, device="cuda")
    buf[shift:shift + xq.nbytes] = torch.from_numpy(xq.reshape(-1)).cuda()
    ys = []
    for x in (dev(xq), buf[shift:shift + xq.nbytes]):
        y = torch.full((m, n), float("nan"), device="cuda")
        getattr(q, "plm_gemm_%s" % fmt)(wd, x, y, m, n, k)
        ys.append(host(y))
    np.testing.assert_array_equal(ys[0], ys[1])
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    assert_close(ys[1], ref, S)


@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
def test_gemm_agrees_with_gemv_small_m(fmt):
    n, k = 96, 1024
    w = make_weights(fmt, 14, 0, n, k)
    for m in (1, 5, 8):
        xq = oracle.quantize_q8K(gen.normal_f32(14, m, m, k))
        a = gpu_matmul("gemm", fmt, w, xq, m, n, k)
        b = gpu_matmul("gemv", fmt, w, xq, m, n, k)
        ref, S = oracle_ref(fmt, w, xq, m, n, k)
        assert_close(a, ref, S)
        assert_close(b, ref, S)


# ------------------------------------------------------- grouped GEMV

@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
@pytest.mark.parametrize("m", [1, 3, 8])
def test_grouped_gemv_equals_single_calls(fmt, m):
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import dev
    shapes = [(40, 1024), (7, 256), (130, 2048), (33, 3072), (1, 1280), (64, 512)]
    probs, want = [], []
    for j, (n, k) in enumerate(shapes):
        w = make_weights(fmt, 20 + j, 0, n, k)
        xq = oracle.quantize_q8K(gen.normal_f32(20 + j, m, m, k))
        ref, S = oracle_ref(fmt, w, xq, m, n, k)
        single = gpu_matmul("gemv", fmt, w, xq, m, n, k)
        assert_close(single, ref, S)
        wd, xd = dev(w), dev(xq)
        y = torch.full((m, n), float("nan"), device="cuda")
        probs.append((wd, xd, y, n, k))
        want.append(single)
    getattr(q, "plm_gemv_%s_grouped" % fmt)(probs, m)
    torch.cuda.synchronize()
    for (_, _, y, _, _), single in zip(probs, want):
        np.testing.assert_array_equal(y.cpu().numpy(), single)


def test_no_device_fault_recorded():
    import quant_packed_gemv_gb300 as q
    assert q.plm_device_fault() == 0


@pytest.mark.parametrize("fmt", ["q2K", "q3K", "q4K", "q5K", "q6K"])
def test_gemm_with_caller_workspace_matches(fmt):
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import dev
    m, n, k = 150, 260, 2048
    w = make_weights(fmt, 30, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(30, 1, m, k))
    # the split-K workspace (here two splits): the same bits as the plain entry,
    # which widens the activation codes in the kernel instead of a pre-pass and
    # splits K the same way over a thread-block cluster, adding the partials
    # in the same order
    full = q.plm_gemm_workspace_size_split(fmt, m, n, k)
    wsf = torch.empty(max(full, 1), dtype=torch.uint8, device="cuda")
    yf = torch.full((m, n), float("nan"), device="cuda")
    getattr(q, "plm_gemm_%s_ws" % fmt)(dev(w), dev(xq), yf, m, n, k, wsf if full else None, full)
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    assert_close(host(yf), ref, S)
    assert np.array_equal(host(yf), gpu_matmul("gemm", fmt, w, xq, m, n, k))
    # the minimal workspace: unsplit, within tolerance
    need = q.plm_gemm_workspace_size(fmt, m, k)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    y = torch.full((m, n), float("nan"), device="cuda")
    getattr(q, "plm_gemm_%s_ws" % fmt)(dev(w), dev(xq), y, m, n, k, ws if need else None, need)
    assert_close(host(y), ref, S)
    if need:
        from quant_packed_gemv_gb300 import plm as P
        small = P.raw_status("plm_gemm_%s_ws" % fmt, dev(w).data_ptr(), dev(xq).data_ptr(), y.data_ptr(),
                             m, n, k, ws.data_ptr(), need - 1, None)
        assert small == P.PLM_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["q4K", "q5K", "q6K"])
@pytest.mark.parametrize("m,n,k", [(64, 256, 4096), (9, 130, 8192), (200, 300, 12288)])
def test_gemm_split_k(fmt, m, n, k):
    """Few output tiles: with the larger workspace the GEMM splits K and adds
    the splits in a fixed order; with the minimal one it does not split.  Both
    match the oracle, and the split result repeats bit for bit."""
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import dev, host
    w = make_weights(fmt, 40, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(40, 2, m, k))
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    wd, xd = dev(w), dev(xq)
    big, small = q.plm_gemm_workspace_size_split(fmt, m, n, k), q.plm_gemm_workspace_size(fmt, m, k)
    assert big > small > 0
    outs = []
    for need in (big, big, small):
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        y = torch.full((m, n), float("nan"), device="cuda")
        getattr(q, "plm_gemm_%s_ws" % fmt)(wd, xd, y, m, n, k, ws, need)
        outs.append(host(y))
        assert_close(outs[-1], ref, S)
    np.testing.assert_array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", ["q2K", "q4K", "q6K"])
def test_gemm_short_last_wave(fmt):
    """More output tiles than SMs with a short last wave: 640 x 4096 gives
    5 x 32 = 160 tiles on 152 SMs, so the last weight-tile rows run as a
    second launch with K split over a cluster.  Every element matches the
    oracle in both entry forms, which give the same bits, run after run."""
    import torch
    import quant_packed_gemv_gb300 as q
    from tests.gpu_helpers import dev, host
    m, n, k = 640, 4096, 2048
    w = make_weights(fmt, 41, 0, n, k)
    xq = oracle.quantize_q8K(gen.normal_f32(41, 3, m, k))
    ref, S = oracle_ref(fmt, w, xq, m, n, k)
    wd, xd = dev(w), dev(xq)
    need = q.plm_gemm_workspace_size_split(fmt, m, n, k)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    outs = []
    for form in ("ws", "ws", "plain"):
        y = torch.full((m, n), float("nan"), device="cuda")
        if form == "ws":
            getattr(q, "plm_gemm_%s_ws" % fmt)(wd, xd, y, m, n, k, ws, need)
        else:
            getattr(q, "plm_gemm_%s" % fmt)(wd, xd, y, m, n, k)
        outs.append(host(y))
        assert_close(outs[-1], ref, S)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])
    assert q.plm_device_fault() == 0
