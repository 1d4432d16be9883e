"""Helpers for the GPU parity tests: move generated inputs to the device,
run the library through its C ABI, and compare with the oracle."""
import numpy as np
import torch

import gen
import oracle
import quant_packed_gemv_gb300 as q

TOL = 1e-4  # max |y_gpu - y_f64| relative to sum_k |w_hat * x_hat|


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def make_weights(fmt, seed, stream, n, k):
    return getattr(gen, "%s_blocks" % fmt)(seed, stream, n, k)


def gpu_quantize(x_np):
    m, k = x_np.shape
    x = dev(x_np)
    xq = torch.empty((m, k // 256 * 292), dtype=torch.uint8, device="cuda")
    q.plm_quantize_q8K(x, xq, m, k)
    return xq


def gpu_matmul(kind, fmt, w_np, xq_np, m, n, k, poison=True):
    """kind: 'gemv' or 'gemm'. Returns y as numpy f32 [m, n]; y is NaN-filled
    first and guarded by trailing canary words."""
    w, xq = dev(w_np), dev(xq_np)
    guard = 64
    ybuf = torch.full((m * n + guard,), float("nan") if poison else 0.0, dtype=torch.float32, device="cuda")
    ybuf[m * n:] = 12345.0
    fn = getattr(q, "plm_%s_%s" % (kind, fmt))
    fn(w, xq, ybuf, m, n, k)
    out = host(ybuf)
    assert np.all(out[m * n:] == 12345.0), "write past the end of y"
    y = out[:m * n].reshape(m, n)
    assert not np.isnan(y).any(), "unwritten output elements"
    return y


def gpu_subdots(fmt, w_np, xq_np, m, n, k):
    per = 8 if fmt in ("q4K", "q5K") else 16   # 32-weight sub-blocks or 16-weight groups
    w, xq = dev(w_np), dev(xq_np)
    out = torch.full((m, n, k // 256 * per), -7, dtype=torch.int32, device="cuda")
    getattr(q, "plm_subdots_%s" % fmt)(w, xq, out, m, n, k)
    return host(out)


def oracle_ref(fmt, w_np, xq_np, m, n, k):
    return (getattr(oracle, "gemm_%s_f64" % fmt)(w_np, xq_np, m, n, k),
            getattr(oracle, "absscale_%s" % fmt)(w_np, xq_np, m, n, k))


def assert_close(y, ref, S, tol=TOL):
    err = np.abs(y.astype(np.float64) - ref)
    bad = err > tol * S
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%d elements out of tolerance; first at %s: got %r want %r (S=%r)"
                             % (bad.sum(), tuple(i), y[tuple(i)], ref[tuple(i)], S[tuple(i)]))
    return float((err / np.maximum(S, 1e-300)).max())
