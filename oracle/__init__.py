"""ORACLE -- test infrastructure, not product code.

Plain scalar C (``plm_ref.c``) wrapped with ctypes and numpy.  It states what
the PocketLLM pages' packed-weight matmul ``gemm_quant`` computes (q8_K
activation quantization, q4_K / q6_K block decode, integer sub-block dots,
the f64 and f32 block combine) so that the CUDA library can be checked
against it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU
baseline leg may import this package; the product path never does, and the
two share no code.

Every function is pinned by a host test against something other than itself
(closed forms, brute force, an independent dequantize-then-matmul in f64, the
exhaustive numpy binary16 decode); none is "parity unpinned".
"""
import ctypes
import fcntl
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "plm_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libplmref.so")

QK = 256
Q4K_BYTES = 144
Q5K_BYTES = 176
Q2K_BYTES = 84
Q3K_BYTES = 110
Q6K_BYTES = 210
Q8K_BYTES = 292

_lib = None


def build(force=False):
    """Compile plm_ref.c (gcc -O2 -ffp-contract=off, OpenMP row loops)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    with open(os.path.join(_OUT_DIR, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=gnu99", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        sig6 = [vp, vp, vp, i64, i64, i64]
        for name in ("plm_ref_subdots_q4K", "plm_ref_subdots_q5K", "plm_ref_subdots_q6K",
                     "plm_ref_gemm_q5K_f64", "plm_ref_gemm_q5K_f32", "plm_ref_absscale_q5K",
                     "plm_ref_subdots_q2K", "plm_ref_gemm_q2K_f64", "plm_ref_gemm_q2K_f32", "plm_ref_absscale_q2K",
                     "plm_ref_subdots_q3K", "plm_ref_gemm_q3K_f64", "plm_ref_gemm_q3K_f32", "plm_ref_absscale_q3K",
                     "plm_ref_gemm_q4K_f64", "plm_ref_gemm_q4K_f32",
                     "plm_ref_gemm_q6K_f64", "plm_ref_gemm_q6K_f32",
                     "plm_ref_absscale_q4K", "plm_ref_absscale_q6K"):
            getattr(lib, name).argtypes = sig6
            getattr(lib, name).restype = None
        for name in ("plm_ref_dequant_q2K", "plm_ref_dequant_q3K", "plm_ref_dequant_q4K", "plm_ref_dequant_q5K",
                     "plm_ref_dequant_q6K", "plm_ref_dequant_q8K", "plm_ref_dequant_q4K_x16",
                     "plm_ref_dequant_q6K_x16"):
            getattr(lib, name).argtypes = [vp, vp, i64, i64]
            getattr(lib, name).restype = None
        lib.plm_ref_quantize_q8K.argtypes = [vp, vp, i64, i64]
        lib.plm_ref_quantize_q8K.restype = None
        lib.plm_ref_f16_array.argtypes = [vp, vp, i64]
        lib.plm_ref_f16_array.restype = None
        lib.plm_ref_q4K_scale_min.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                              ctypes.POINTER(ctypes.c_int)]
        lib.plm_ref_q4K_scale_min.restype = None
        lib.plm_ref_q3K_scale.argtypes = [vp, ctypes.c_int]
        lib.plm_ref_q3K_scale.restype = ctypes.c_int
        lib.plm_ref_swiglu_f64.argtypes = [vp, vp, vp, i64]
        lib.plm_ref_swiglu_f64.restype = None
        lib.plm_ref_set_threads.argtypes = [ctypes.c_int]
        lib.plm_ref_set_threads.restype = None
        lib.plm_ref_max_threads.argtypes = []
        lib.plm_ref_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a):
    assert a.flags.c_contiguous
    return ctypes.c_void_p(a.ctypes.data)


def _u8(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8
    return a


def set_threads(t):
    _load().plm_ref_set_threads(int(t))


def max_threads():
    return _load().plm_ref_max_threads()


def f16_to_f32(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().plm_ref_f16_array(_p(bits), _p(out), bits.size)
    return out


def quantize_q8K(x):
    """x: float32 [m, k] -> q8_K bytes uint8 [m, k/256*292]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    m, k = x.shape
    assert k % QK == 0
    out = np.empty((m, k // QK * Q8K_BYTES), dtype=np.uint8)
    _load().plm_ref_quantize_q8K(_p(x), _p(out), m, k)
    return out


def q4K_scale_min(table12, j):
    t = np.ascontiguousarray(table12, dtype=np.uint8)
    assert t.size == 12
    sc, mn = ctypes.c_int(), ctypes.c_int()
    _load().plm_ref_q4K_scale_min(_p(t), int(j), ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def _call6(name, w, xq, m, n, k, shape, dtype):
    w, xq = _u8(w), _u8(xq)
    out = np.empty(shape, dtype=dtype)
    getattr(_load(), name)(_p(w), _p(xq), _p(out), m, n, k)
    return out


def subdots_q4K(w, xq, m, n, k):
    """int32 [m, n, k/256*8]: per 32-weight sub-block integer dots."""
    return _call6("plm_ref_subdots_q4K", w, xq, m, n, k, (m, n, k // QK * 8), np.int32)


def _dequant(name, w, n, k):
    w = _u8(w)
    out = np.empty((n, k), dtype=np.float64)
    getattr(_load(), name)(_p(w), _p(out), n, k)
    return out


def subdots_q2K(w, xq, m, n, k):
    return _call6("plm_ref_subdots_q2K", w, xq, m, n, k, (m, n, k // 16), np.int32)


def subdots_q3K(w, xq, m, n, k):
    return _call6("plm_ref_subdots_q3K", w, xq, m, n, k, (m, n, k // 16), np.int32)


def gemm_q2K_f64(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q2K_f64", w, xq, m, n, k, (m, n), np.float64)


def gemm_q2K_f32(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q2K_f32", w, xq, m, n, k, (m, n), np.float32)


def gemm_q3K_f64(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q3K_f64", w, xq, m, n, k, (m, n), np.float64)


def gemm_q3K_f32(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q3K_f32", w, xq, m, n, k, (m, n), np.float32)


def absscale_q2K(w, xq, m, n, k):
    return _call6("plm_ref_absscale_q2K", w, xq, m, n, k, (m, n), np.float64)


def absscale_q3K(w, xq, m, n, k):
    return _call6("plm_ref_absscale_q3K", w, xq, m, n, k, (m, n), np.float64)


def dequant_q2K(w, n, k):
    return _dequant("plm_ref_dequant_q2K", w, n, k)


def dequant_q3K(w, n, k):
    return _dequant("plm_ref_dequant_q3K", w, n, k)


def q3K_scale(table12, g):
    t = _u8(np.asarray(table12, dtype=np.uint8))
    return _load().plm_ref_q3K_scale(_p(t), g)


def subdots_q5K(w, xq, m, n, k):
    return _call6("plm_ref_subdots_q5K", w, xq, m, n, k, (m, n, k // 32), np.int32)


def gemm_q5K_f64(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q5K_f64", w, xq, m, n, k, (m, n), np.float64)


def gemm_q5K_f32(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q5K_f32", w, xq, m, n, k, (m, n), np.float32)


def absscale_q5K(w, xq, m, n, k):
    return _call6("plm_ref_absscale_q5K", w, xq, m, n, k, (m, n), np.float64)


def dequant_q5K(w, n, k):
    w = _u8(w)
    out = np.empty((n, k), dtype=np.float64)
    _load().plm_ref_dequant_q5K(_p(w), _p(out), n, k)
    return out


def subdots_q6K(w, xq, m, n, k):
    """int32 [m, n, k/256*16]: per 16-weight group integer dots (q6 - 32)."""
    return _call6("plm_ref_subdots_q6K", w, xq, m, n, k, (m, n, k // QK * 16), np.int32)


def gemm_q4K_f64(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q4K_f64", w, xq, m, n, k, (m, n), np.float64)


def gemm_q4K_f32(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q4K_f32", w, xq, m, n, k, (m, n), np.float32)


def gemm_q6K_f64(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q6K_f64", w, xq, m, n, k, (m, n), np.float64)


def gemm_q6K_f32(w, xq, m, n, k):
    return _call6("plm_ref_gemm_q6K_f32", w, xq, m, n, k, (m, n), np.float32)


def swiglu_f64(g, u):
    """h = silu(g) * u elementwise in f64 (the gate/up pair's epilogue)."""
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert g.shape == u.shape
    h = np.empty_like(g)
    _load().plm_ref_swiglu_f64(_p(g), _p(u), _p(h), g.size)
    return h


def swiglu_q4K_f64(w_gate, w_up, xq, m, n, k):
    """h = silu(W_gate . x) * (W_up . x) in f64 on the oracle's integer path."""
    return swiglu_f64(gemm_q4K_f64(w_gate, xq, m, n, k), gemm_q4K_f64(w_up, xq, m, n, k))


def absscale_q4K(w, xq, m, n, k):
    return _call6("plm_ref_absscale_q4K", w, xq, m, n, k, (m, n), np.float64)


def absscale_q6K(w, xq, m, n, k):
    return _call6("plm_ref_absscale_q6K", w, xq, m, n, k, (m, n), np.float64)


def dequant_q4K(w, n, k):
    w = _u8(w)
    out = np.empty((n, k), dtype=np.float64)
    _load().plm_ref_dequant_q4K(_p(w), _p(out), n, k)
    return out


def dequant_q4K_x16(wx, n, k):
    """f64 weights [n, k] read from the row-interleaved x16 layout (the q4_K
    blocks of 16-row tiles, 16-byte units permuted; see plm_ref.c)."""
    wx = _u8(wx)
    out = np.empty((n, k), dtype=np.float64)
    _load().plm_ref_dequant_q4K_x16(_p(wx), _p(out), n, k)
    return out


def dequant_q6K_x16(wx, n, k):
    """f64 weights [n, k] read from the x16 layout of q6_K (see plm_ref.c)."""
    wx = _u8(wx)
    out = np.empty((n, k), dtype=np.float64)
    _load().plm_ref_dequant_q6K_x16(_p(wx), _p(out), n, k)
    return out


def dequant_q6K(w, n, k):
    w = _u8(w)
    out = np.empty((n, k), dtype=np.float64)
    _load().plm_ref_dequant_q6K(_p(w), _p(out), n, k)
    return out


def dequant_q8K(xq, m, k):
    xq = _u8(xq)
    out = np.empty((m, k), dtype=np.float64)
    _load().plm_ref_dequant_q8K(_p(xq), _p(out), m, k)
    return out


Q8K_DTYPE = np.dtype([("d", "<f4"), ("qs", "i1", (256,)), ("bsums", "<i2", (16,))])


def q8K_fields(xq, m, k):
    """View q8_K bytes as a structured array [m, k/256] with d, qs, bsums."""
    return np.ascontiguousarray(xq).view(Q8K_DTYPE).reshape(m, k // QK)
