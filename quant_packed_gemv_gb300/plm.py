"""Python binding of libplm: the C ABI of include/plm.h, same names.

Argument marshalling only.  Device buffers are torch tensors (or raw integer
device addresses); the stream is a torch.cuda.Stream, a raw cudaStream_t
integer, or None for torch's current stream.  Every computation runs in the
library's CUDA kernels; there is no host or library fallback, and loading
fails loudly when libplm.so is missing.
"""
import ctypes
import os

from . import build as _build

PLM_OK = 0
PLM_ERR_INVALID_ARG = 1
PLM_ERR_MISALIGNED = 2
PLM_ERR_UNSUPPORTED = 3
PLM_ERR_CUDA = 4

QK = 256
Q4K_BYTES = 144
Q5K_BYTES = 176
Q2K_BYTES = 84
Q3K_BYTES = 110
Q6K_BYTES = 210
Q8K_BYTES = 292
GEMV_MAX_M = 8
PLM_NOALLOC_WORKSPACE_BYTES = 32 << 20   # the fixed array of plm_gemm_q4K_noalloc


class PlmError(RuntimeError):
    def __init__(self, fn, status, lib):
        self.status = status
        msg = lib.plm_status_string(status).decode()
        if status == PLM_ERR_CUDA:
            msg += " (cudaError %d)" % lib.plm_last_cuda_error()
        super().__init__("%s: %s" % (fn, msg))


class _Problem(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("xq", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


class _SProblem(ctypes.Structure):
    _fields_ = [("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("xq", ctypes.c_void_p),
                ("h", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


class _QProblem(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


_lib = None


def library_path():
    return _build.LIB


def load(build_if_missing=True):
    """Loads libplm.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libplm.so not found at %s; run quant_packed_gemv_gb300.build" % path)
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.plm_abi_version.argtypes = []
    lib.plm_abi_version.restype = ctypes.c_int
    lib.plm_set_overlap.argtypes = [ctypes.c_int]
    lib.plm_set_overlap.restype = ctypes.c_int
    lib.plm_status_string.argtypes = [ctypes.c_int]
    lib.plm_status_string.restype = ctypes.c_char_p
    lib.plm_last_cuda_error.argtypes = []
    lib.plm_last_cuda_error.restype = ctypes.c_int
    lib.plm_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.plm_device_fault.restype = ctypes.c_int
    lib.plm_probe_mma_rates.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    lib.plm_probe_mma_rates.restype = ctypes.c_int
    lib.plm_probe_tcgen05_rate.argtypes = [ctypes.POINTER(ctypes.c_double)] * 3
    lib.plm_probe_tcgen05_rate.restype = ctypes.c_int
    lib.plm_selftest_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.c_int, vp]
    lib.plm_selftest_bounded_wait.restype = ctypes.c_int
    for f in ("q4K", "q6K"):
        getattr(lib, "plm_%s_x16_size" % f).argtypes = [i64, i64]
        getattr(lib, "plm_%s_x16_size" % f).restype = ctypes.c_size_t
        getattr(lib, "plm_%s_to_x16" % f).argtypes = [vp, vp, i64, i64, vp]
        getattr(lib, "plm_%s_to_x16" % f).restype = ctypes.c_int
    lib.plm_quantize_q8K.argtypes = [vp, vp, i64, i64, vp]
    lib.plm_quantize_q8K.restype = ctypes.c_int
    lib.plm_gemm_workspace_size.argtypes = [ctypes.c_int, i64, i64]
    lib.plm_gemm_workspace_size.restype = ctypes.c_size_t
    lib.plm_gemm_workspace_size_split.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.plm_gemm_workspace_size_split.restype = ctypes.c_size_t
    for name in ("plm_gemm_q2K_ws", "plm_gemm_q3K_ws", "plm_gemm_q4K_ws", "plm_gemm_q5K_ws", "plm_gemm_q6K_ws"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, vp, i64, i64, i64, vp, ctypes.c_size_t, vp]
        fn.restype = ctypes.c_int
    for name in ("plm_gemv_q2K_grouped", "plm_gemv_q3K_grouped", "plm_gemv_q4K_grouped", "plm_gemv_q5K_grouped",
                 "plm_gemv_q6K_grouped"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.POINTER(_Problem), i64, i64, vp]
        fn.restype = ctypes.c_int
    lib.plm_gemv_q4K_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.plm_gemv_q4K_swiglu.restype = ctypes.c_int
    lib.plm_gemv_q4K_swiglu_grouped.argtypes = [ctypes.POINTER(_SProblem), i64, i64, vp]
    lib.plm_gemv_q4K_swiglu_grouped.restype = ctypes.c_int
    lib.plm_gemm_q4K_swiglu.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.plm_gemm_q4K_swiglu.restype = ctypes.c_int
    lib.plm_gemm_q4K_swiglu_ws.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, ctypes.c_size_t, vp]
    lib.plm_gemm_q4K_swiglu_ws.restype = ctypes.c_int
    lib.plm_gemm_swiglu_workspace_size.argtypes = [i64, i64, i64]
    lib.plm_gemm_swiglu_workspace_size.restype = ctypes.c_size_t
    lib.plm_quantize_gemv_q4K_grouped.argtypes = [ctypes.POINTER(_QProblem), i64, i64, vp]
    lib.plm_quantize_gemv_q4K_grouped.restype = ctypes.c_int
    for name in ("plm_gemv_q4K", "plm_gemv_q6K", "plm_gemm_q4K", "plm_gemm_q6K", "plm_gemm_q4K_noalloc",
                 "plm_subdots_q4K", "plm_subdots_q6K", "plm_quantize_gemv_q4K",
                 "plm_gemv_q5K", "plm_gemm_q5K", "plm_subdots_q5K",
                 "plm_gemv_q2K", "plm_gemm_q2K", "plm_subdots_q2K", "plm_gemv_q3K", "plm_gemm_q3K", "plm_subdots_q3K",
                 "plm_gemv_q4K_x16", "plm_gemv_q6K_x16"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _addr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, status):
    if status != PLM_OK:
        raise PlmError(fn, status, _lib)


def plm_abi_version():
    return load().plm_abi_version()


PLM_OVERLAP_OFF, PLM_OVERLAP_LAUNCH, PLM_OVERLAP_PREFETCH = 0, 1, 2


def plm_set_overlap(mode):
    """Early-launch mode for later launches (PLM_OVERLAP_*); returns the previous mode."""
    lib = load()
    r = lib.plm_set_overlap(int(mode))
    if r < 0:
        raise PlmError("plm_set_overlap", -r, lib)
    return r


def plm_device_fault(clear=True):
    """Reads (and by default clears) the device fault word; synchronizes."""
    lib = load()
    code = ctypes.c_uint32(0)
    _check("plm_device_fault", lib.plm_device_fault(ctypes.byref(code), 1 if clear else 0))
    return code.value


def plm_selftest_bounded_wait(rounds, complete, stream=None):
    """Launches the bounded-wait self-test (see include/plm.h); asynchronous."""
    lib = load()
    _check("plm_selftest_bounded_wait", lib.plm_selftest_bounded_wait(int(rounds), 1 if complete else 0,
                                                                      _stream(stream)))


def plm_probe_mma_rates():
    """(mma.sync s8 TOPS, mma.sync f16 TFLOPS) measured on the current device; synchronizes."""
    lib = load()
    a, b = ctypes.c_double(0), ctypes.c_double(0)
    _check("plm_probe_mma_rates", lib.plm_probe_mma_rates(ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def plm_probe_tcgen05_rate():
    """(cycles per MMA, cycles per MMA with an mbarrier wait after each commit, TFLOPS on every
    SM) of the GEMM's tcgen05 MMA on the current device; synchronizes."""
    lib = load()
    a, b, c = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    _check("plm_probe_tcgen05_rate", lib.plm_probe_tcgen05_rate(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def plm_quantize_q8K(x, xq, m, k, stream=None):
    lib = load()
    _check("plm_quantize_q8K", lib.plm_quantize_q8K(_addr(x), _addr(xq), m, k, _stream(stream)))


def _mm(name):
    def call(w, xq, y, m, n, k, stream=None):
        lib = load()
        _check(name, getattr(lib, name)(_addr(w), _addr(xq), _addr(y), m, n, k, _stream(stream)))
    call.__name__ = name
    call.__doc__ = "Binding of the C entry point %s(w, xq, out, m, n, k, stream)." % name
    return call


plm_gemv_q4K = _mm("plm_gemv_q4K")
plm_gemv_q6K = _mm("plm_gemv_q6K")
plm_gemv_q5K = _mm("plm_gemv_q5K")
plm_gemm_q5K = _mm("plm_gemm_q5K")
plm_subdots_q5K = _mm("plm_subdots_q5K")
plm_gemv_q2K = _mm("plm_gemv_q2K")
plm_gemm_q2K = _mm("plm_gemm_q2K")
plm_subdots_q2K = _mm("plm_subdots_q2K")
plm_gemv_q3K = _mm("plm_gemv_q3K")
plm_gemm_q3K = _mm("plm_gemm_q3K")
plm_subdots_q3K = _mm("plm_subdots_q3K")
plm_gemm_q4K = _mm("plm_gemm_q4K")
plm_gemm_q6K = _mm("plm_gemm_q6K")
# q4_K GEMM whose workspace is a fixed array inside the library: for callers
# that must not allocate device memory while running (see include/plm.h).
plm_gemm_q4K_noalloc = _mm("plm_gemm_q4K_noalloc")
plm_subdots_q4K = _mm("plm_subdots_q4K")
# fused q8_K producer: f32 activations x in place of xq
plm_quantize_gemv_q4K = _mm("plm_quantize_gemv_q4K")
plm_subdots_q6K = _mm("plm_subdots_q6K")


plm_gemv_q4K_x16 = _mm("plm_gemv_q4K_x16")
plm_gemv_q6K_x16 = _mm("plm_gemv_q6K_x16")


def plm_q4K_x16_size(n, k):
    """Bytes of the row-interleaved x16 form of an n x k q4_K matrix (0: invalid)."""
    return load().plm_q4K_x16_size(n, k)


def plm_q6K_x16_size(n, k):
    """Bytes of the row-interleaved x16 form of an n x k q6_K matrix (0: invalid)."""
    return load().plm_q6K_x16_size(n, k)


def plm_q4K_to_x16(w, w_x16, n, k, stream=None):
    """Repacks q4_K weights into the x16 layout (see include/plm.h)."""
    lib = load()
    _check("plm_q4K_to_x16", lib.plm_q4K_to_x16(_addr(w), _addr(w_x16), n, k, _stream(stream)))


def plm_q6K_to_x16(w, w_x16, n, k, stream=None):
    """Repacks q6_K weights into the x16 layout (see include/plm.h)."""
    lib = load()
    _check("plm_q6K_to_x16", lib.plm_q6K_to_x16(_addr(w), _addr(w_x16), n, k, _stream(stream)))


def _grouped(name):
    def call(problems, m, stream=None):
        """problems: sequence of (w, xq, y, n, k) with device tensors or addresses."""
        lib = load()
        arr = (_Problem * len(problems))()
        for j, (w, xq, y, n, k) in enumerate(problems):
            arr[j] = _Problem(_addr(w), _addr(xq), _addr(y), n, k)
        _check(name, getattr(lib, name)(arr, len(problems), m, _stream(stream)))
    call.__name__ = name
    call.__doc__ = "Binding of %s(problems, count, m, stream)." % name
    return call


plm_gemv_q4K_grouped = _grouped("plm_gemv_q4K_grouped")
plm_gemv_q6K_grouped = _grouped("plm_gemv_q6K_grouped")
plm_gemv_q5K_grouped = _grouped("plm_gemv_q5K_grouped")
plm_gemv_q2K_grouped = _grouped("plm_gemv_q2K_grouped")
plm_gemv_q3K_grouped = _grouped("plm_gemv_q3K_grouped")


def plm_gemv_q4K_swiglu(w_gate, w_up, xq, h, m, n, k, stream=None):
    """h = silu(W_gate . x) * (W_up . x) (see include/plm.h)."""
    lib = load()
    _check("plm_gemv_q4K_swiglu", lib.plm_gemv_q4K_swiglu(_addr(w_gate), _addr(w_up), _addr(xq), _addr(h), m, n, k,
                                                          _stream(stream)))


def plm_gemm_swiglu_workspace_size(m, n, k):
    """Workspace bytes of plm_gemm_q4K_swiglu_ws (0: none needed, or invalid arguments)."""
    return load().plm_gemm_swiglu_workspace_size(m, n, k)


def plm_gemm_q4K_swiglu(w_gate, w_up, xq, h, m, n, k, stream=None):
    """Prefill gate/up pair: h = silu(W_gate . x) * (W_up . x) (see include/plm.h)."""
    lib = load()
    _check("plm_gemm_q4K_swiglu", lib.plm_gemm_q4K_swiglu(_addr(w_gate), _addr(w_up), _addr(xq), _addr(h), m, n, k,
                                                          _stream(stream)))


def plm_gemm_q4K_swiglu_ws(w_gate, w_up, xq, h, m, n, k, workspace, workspace_bytes=None, stream=None):
    """plm_gemm_q4K_swiglu with a caller-owned workspace (plm_gemm_swiglu_workspace_size bytes)."""
    lib = load()
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("plm_gemm_q4K_swiglu_ws", lib.plm_gemm_q4K_swiglu_ws(_addr(w_gate), _addr(w_up), _addr(xq), _addr(h), m,
                                                                n, k, _addr(workspace), workspace_bytes,
                                                                _stream(stream)))


def plm_gemv_q4K_swiglu_grouped(problems, m, stream=None):
    """problems: sequence of (w_gate, w_up, xq, h, n, k) with device tensors or addresses."""
    lib = load()
    arr = (_SProblem * len(problems))()
    for j, (wg, wu, xq, h, n, k) in enumerate(problems):
        arr[j] = _SProblem(_addr(wg), _addr(wu), _addr(xq), _addr(h), n, k)
    _check("plm_gemv_q4K_swiglu_grouped", lib.plm_gemv_q4K_swiglu_grouped(arr, len(problems), m, _stream(stream)))


def plm_quantize_gemv_q4K_grouped(problems, m, stream=None):
    """problems: sequence of (w, x_f32, y, n, k) with device tensors or addresses."""
    lib = load()
    arr = (_QProblem * len(problems))()
    for j, (w, x, y, n, k) in enumerate(problems):
        arr[j] = _QProblem(_addr(w), _addr(x), _addr(y), n, k)
    _check("plm_quantize_gemv_q4K_grouped", lib.plm_quantize_gemv_q4K_grouped(arr, len(problems), m, _stream(stream)))


def plm_gemm_workspace_size(fmt, m, k):
    """fmt: 'q2K' .. 'q6K' or 2 .. 6."""
    f = {"q2K": 2, "q3K": 3, "q4K": 4, "q5K": 5, "q6K": 6}.get(fmt, fmt)
    return load().plm_gemm_workspace_size(f, m, k)


def plm_gemm_workspace_size_split(fmt, m, n, k):
    """Workspace bytes that let the GEMM split K (see include/plm.h)."""
    f = {"q2K": 2, "q3K": 3, "q4K": 4, "q5K": 5, "q6K": 6}.get(fmt, fmt)
    return load().plm_gemm_workspace_size_split(f, m, n, k)


def _gemm_ws(name):
    def call(w, xq, y, m, n, k, workspace, workspace_bytes=None, stream=None):
        lib = load()
        if workspace_bytes is None:
            workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(name, getattr(lib, name)(_addr(w), _addr(xq), _addr(y), m, n, k, _addr(workspace),
                                        workspace_bytes, _stream(stream)))
    call.__name__ = name
    call.__doc__ = "Binding of %s(w, xq, y, m, n, k, workspace, bytes, stream)." % name
    return call


plm_gemm_q4K_ws = _gemm_ws("plm_gemm_q4K_ws")
plm_gemm_q6K_ws = _gemm_ws("plm_gemm_q6K_ws")
plm_gemm_q5K_ws = _gemm_ws("plm_gemm_q5K_ws")
plm_gemm_q2K_ws = _gemm_ws("plm_gemm_q2K_ws")
plm_gemm_q3K_ws = _gemm_ws("plm_gemm_q3K_ws")


def raw_status(name, *args):
    """Calls an entry point and returns its status code without raising
    (used by the argument-check tests)."""
    return getattr(load(), name)(*args)
