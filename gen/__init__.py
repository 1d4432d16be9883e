"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

The C source ``plmgen.c`` beside this file documents the draw layout.  This
module compiles it on first use (gcc, in-tree ``_build/``) and wraps it with
numpy.  It holds none of the packed-matmul arithmetic: it fills block fields
with random values and nothing else.
"""
import ctypes
import fcntl
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "plmgen.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libplmgen.so")

Q4K_BYTES = 144
Q5K_BYTES = 176
Q2K_BYTES = 84
Q3K_BYTES = 110
Q6K_BYTES = 210
QK = 256

_lib = None


def build(force=False):
    """Compile plmgen.c into _build/libplmgen.so (idempotent, process-safe)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    with open(os.path.join(_OUT_DIR, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        for name in ("plmgen_q2K", "plmgen_q3K", "plmgen_q4K", "plmgen_q5K", "plmgen_q6K", "plmgen_normal_f32",
                     "plmgen_raw"):
            fn = getattr(lib, name)
            fn.argtypes = [u64, u64, i64, i64, vp]
            fn.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def q4K_blocks(seed, stream, n, k, row0=0, out=None):
    """Rows [row0, row0+n) of an n_total x k q4_K matrix as uint8 [n, k/256*144]."""
    assert k % QK == 0
    nb = k // QK
    if out is None:
        out = np.empty((n, nb * Q4K_BYTES), dtype=np.uint8)
    assert out.flags.c_contiguous and out.nbytes == n * nb * Q4K_BYTES
    _load().plmgen_q4K(seed, stream, row0 * nb, n * nb, _ptr(out))
    return out


def _blocks(fn, bpb, seed, stream, n, k, row0, out):
    assert k % QK == 0
    nb = k // QK
    if out is None:
        out = np.empty((n, nb * bpb), dtype=np.uint8)
    assert out.flags.c_contiguous and out.nbytes == n * nb * bpb
    getattr(_load(), fn)(seed, stream, row0 * nb, n * nb, _ptr(out))
    return out


def q2K_blocks(seed, stream, n, k, row0=0, out=None):
    """Rows [row0, row0+n) of a q2_K matrix as uint8 [n, k/256*84]."""
    return _blocks("plmgen_q2K", Q2K_BYTES, seed, stream, n, k, row0, out)


def q3K_blocks(seed, stream, n, k, row0=0, out=None):
    """Rows [row0, row0+n) of a q3_K matrix as uint8 [n, k/256*110]."""
    return _blocks("plmgen_q3K", Q3K_BYTES, seed, stream, n, k, row0, out)


def q5K_blocks(seed, stream, n, k, row0=0, out=None):
    """Rows [row0, row0+n) of a q5_K matrix as uint8 [n, k/256*176]."""
    assert k % QK == 0
    nb = k // QK
    if out is None:
        out = np.empty((n, nb * Q5K_BYTES), dtype=np.uint8)
    assert out.flags.c_contiguous and out.nbytes == n * nb * Q5K_BYTES
    _load().plmgen_q5K(seed, stream, row0 * nb, n * nb, _ptr(out))
    return out


def q6K_blocks(seed, stream, n, k, row0=0, out=None):
    """Rows [row0, row0+n) of a q6_K matrix as uint8 [n, k/256*210]."""
    assert k % QK == 0
    nb = k // QK
    if out is None:
        out = np.empty((n, nb * Q6K_BYTES), dtype=np.uint8)
    assert out.flags.c_contiguous and out.nbytes == n * nb * Q6K_BYTES
    _load().plmgen_q6K(seed, stream, row0 * nb, n * nb, _ptr(out))
    return out


def normal_f32(seed, stream, m, k, out=None):
    """Activations x: float32 [m, k] ~ N(0, 1)."""
    if out is None:
        out = np.empty((m, k), dtype=np.float32)
    assert out.flags.c_contiguous and out.size == m * k
    _load().plmgen_normal_f32(seed, stream, 0, m * k, _ptr(out))
    return out


def raw_draws(seed, stream, first, count):
    out = np.empty(count, dtype=np.uint64)
    _load().plmgen_raw(seed, stream, first, count, _ptr(out))
    return out
