"""Python binding of libgdn.so (the C ABI in include/gdn.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, and their data pointers plus the current CUDA stream go to the C
functions of the same names.  Every step of the computation runs in the CUDA
kernels of libgdn.so; there is no fallback.  If the library has not been built
the first call raises.

PyTorch provides device memory and streams; nothing here computes with it.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_SEQUENTIAL = 0
GDN_CHUNKED = 1
GDN_AUTO = 2
GDN_AUTO_CHUNKED_MIN_T = 64
GDN_OK = 0
GDN_ERR_INVALID_ARG = -1
GDN_ERR_UNSUPPORTED = -2
GDN_ERR_ALLOC = -3
GDN_ERR_CUDA = -4
GDN_ERR_TIMEOUT = -5
# options (gdn_set_option)
GDN_OPT_CHUNK_PRODUCTS = 1
GDN_OPT_CHUNK_ONE_LAUNCH = 2
GDN_OPT_NORM_IN_LAUNCH = 3
GDN_OPT_SEQ_ROWS_PER_THREAD = 4
GDN_OPT_CHUNK_PREP_CTAS = 5
GDN_OPT_TEST_WITHHOLD_PREP_TASK = 101
GDN_OPT_TEST_FAIL_SCRATCH_ALLOC = 102
GDN_PRODUCTS_MMA = 0
GDN_PRODUCTS_FMA = 1
GDN_PRODUCTS_TCGEN05 = 2
GDN_PRODUCTS_TMEM = 3
_OPTIONS = {"chunk_products": GDN_OPT_CHUNK_PRODUCTS, "chunk_one_launch": GDN_OPT_CHUNK_ONE_LAUNCH,
            "norm_in_launch": GDN_OPT_NORM_IN_LAUNCH, "seq_rows_per_thread": GDN_OPT_SEQ_ROWS_PER_THREAD,
            "chunk_prep_ctas": GDN_OPT_CHUNK_PREP_CTAS,
            "test_withhold_prep_task": GDN_OPT_TEST_WITHHOLD_PREP_TASK,
            "test_fail_scratch_alloc": GDN_OPT_TEST_FAIL_SCRATCH_ALLOC}
_PRODUCTS = {"mma": GDN_PRODUCTS_MMA, "fma": GDN_PRODUCTS_FMA, "tc": GDN_PRODUCTS_TCGEN05,
             "tcgen05": GDN_PRODUCTS_TCGEN05, "tmem": GDN_PRODUCTS_TMEM}

_MODES = {"sequential": GDN_SEQUENTIAL, "seq": GDN_SEQUENTIAL, "chunked": GDN_CHUNKED, "auto": GDN_AUTO,
          GDN_SEQUENTIAL: GDN_SEQUENTIAL, GDN_CHUNKED: GDN_CHUNKED, GDN_AUTO: GDN_AUTO}

_lock = threading.Lock()
_lib = None

EXPORTS = ("gdn_recurrence", "gdn_out_norm", "gdn_last_error", "gdn_device_status",
           "gdn_release_scratch", "gdn_poison_scratch", "gdn_chunked_scratch_bytes", "gdn_launch_count",
           "gdn_recurrence_chunked_noalloc", "gdn_decode", "gdn_prestage", "gdn_recurrence_norm",
           "gdn_set_option", "gdn_get_option")


class GDNError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so and declare its C signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run linear_attention_recurrence_gb300.build.build() "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.gdn_recurrence.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp]
        lib.gdn_recurrence.restype = i32
        lib.gdn_recurrence_chunked_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp]
        lib.gdn_recurrence_chunked_noalloc.restype = i32
        lib.gdn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
        lib.gdn_decode.restype = i32
        lib.gdn_prestage.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32,
                                     ctypes.c_float, vp]
        lib.gdn_prestage.restype = i32
        lib.gdn_recurrence_norm.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, i64, i32, i32, i32,
                                            i32, vp]
        lib.gdn_recurrence_norm.restype = i32
        lib.gdn_out_norm.argtypes = [vp, vp, vp, ctypes.c_float, vp, i64, i32, i32, vp]
        lib.gdn_out_norm.restype = i32
        lib.gdn_last_error.argtypes = []
        lib.gdn_last_error.restype = ctypes.c_char_p
        lib.gdn_device_status.argtypes = [vp]
        lib.gdn_device_status.restype = i32
        lib.gdn_release_scratch.argtypes = [i32]
        lib.gdn_release_scratch.restype = i32
        lib.gdn_poison_scratch.argtypes = [ctypes.c_uint32, i32, vp]
        lib.gdn_poison_scratch.restype = i32
        lib.gdn_chunked_scratch_bytes.argtypes = [i32]
        lib.gdn_chunked_scratch_bytes.restype = ctypes.c_size_t
        lib.gdn_set_option.argtypes = [i32, i32]
        lib.gdn_set_option.restype = i32
        lib.gdn_get_option.argtypes = [i32, ctypes.POINTER(ctypes.c_int)]
        lib.gdn_get_option.restype = i32
        lib.gdn_launch_count.argtypes = []
        lib.gdn_launch_count.restype = ctypes.c_uint64
        if path == LIB_PATH:
            _lib = lib
        return lib


def _check(rc: int):
    if rc != GDN_OK:
        raise GDNError(rc, load_library().gdn_last_error().decode(errors="replace"))


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _want(t, name, shape=None, dtype=torch.float32):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def gdn_recurrence(q, k, v, g, beta, state, out=None, mode="sequential", stream=None):
    """Gated delta-rule recurrence; updates ``state`` in place and returns ``out``.

    q, k: [T][n_kh][d]; v: [T][n_vh][d]; g, beta: [T][n_vh]; state: [n_vh][d][d]
    (FP32, CUDA, contiguous).  ``out`` ([T][n_vh][d]) is allocated if None.
    """
    T, n_kh, d = q.shape
    n_vh = v.shape[1]
    _want(q, "q", (T, n_kh, d))
    _want(k, "k", (T, n_kh, d))
    _want(v, "v", (T, n_vh, d))
    _want(g, "g", (T, n_vh))
    _want(beta, "beta", (T, n_vh))
    _want(state, "state", (n_vh, d, d))
    if out is None:
        out = torch.empty((T, n_vh, d), dtype=torch.float32, device=q.device)
    _want(out, "out", (T, n_vh, d))
    if mode not in _MODES:
        raise ValueError(f"unknown mode {mode!r}")
    lib = load_library()
    rc = lib.gdn_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                            T, n_kh, n_vh, d, _MODES[mode], _stream_ptr(stream))
    _check(rc)
    return out


def gdn_recurrence_norm(q, k, v, g, beta, state, z, w, eps: float = 1e-6, out=None, y=None, mode="chunked",
                        stream=None, store_out=True):
    """gdn_recurrence and gdn_out_norm of its output in one call; returns (out, y).

    ``out`` ([T][n_vh][d] FP32) and ``y`` ([T][n_vh][d] float16) are allocated if
    None.  With ``store_out=False`` the FP32 output is not written at all (``out``
    is returned as None): the norm is then fused into the scan, in sequential mode
    and in chunked mode's tensor-memory form (the default); chunked mode's other
    product forms need the FP32 output.
    """
    T, n_kh, d = q.shape
    n_vh = v.shape[1]
    _want(q, "q", (T, n_kh, d))
    _want(k, "k", (T, n_kh, d))
    _want(v, "v", (T, n_vh, d))
    _want(g, "g", (T, n_vh))
    _want(beta, "beta", (T, n_vh))
    _want(state, "state", (n_vh, d, d))
    _want(z, "z", (T, n_vh, d))
    _want(w, "w", (d,))
    if not store_out:
        out = None
    elif out is None:
        out = torch.empty((T, n_vh, d), dtype=torch.float32, device=q.device)
    if y is None:
        y = torch.empty((T, n_vh, d), dtype=torch.float16, device=q.device)
    if out is not None:
        _want(out, "out", (T, n_vh, d))
    _want(y, "y", (T, n_vh, d), dtype=torch.float16)
    if mode not in _MODES:
        raise ValueError(f"unknown mode {mode!r}")
    lib = load_library()
    rc = lib.gdn_recurrence_norm(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out), _ptr(z),
                                 _ptr(w), float(eps), _ptr(y), T, n_kh, n_vh, d, _MODES[mode], _stream_ptr(stream))
    _check(rc)
    return out, y


def gdn_decode(q, k, v, g, beta, states, out=None, stream=None):
    """One decode step for a batch of independent sequences; updates ``states``
    in place and returns ``out``.

    q, k: [B][n_kh][d]; v: [B][n_vh][d]; g, beta: [B][n_vh]; states:
    [B][n_vh][d][d].  ``out`` ([B][n_vh][d]) is allocated if None.
    """
    B, n_kh, d = q.shape
    n_vh = v.shape[1]
    _want(q, "q", (B, n_kh, d))
    _want(k, "k", (B, n_kh, d))
    _want(v, "v", (B, n_vh, d))
    _want(g, "g", (B, n_vh))
    _want(beta, "beta", (B, n_vh))
    _want(states, "states", (B, n_vh, d, d))
    if out is None:
        out = torch.empty((B, n_vh, d), dtype=torch.float32, device=q.device)
    _want(out, "out", (B, n_vh, d))
    lib = load_library()
    rc = lib.gdn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(states), _ptr(out),
                        B, n_kh, n_vh, d, _stream_ptr(stream))
    _check(rc)
    return out


def gdn_prestage(qkv, conv_w, a, b, A_log, dt_bias, n_kh: int, n_vh: int, hist_in=None, hist_out=None,
                 activation: int = 1, eps: float = 1e-6, out=None, stream=None):
    """The pre-stage: q, k, v, g, beta for gdn_recurrence from the packed qkv
    projections (causal 4-tap convolution, optional SiLU, q/k L2 norms, gates).

    qkv: [T][(2 n_kh + n_vh) d]; conv_w: [(2 n_kh + n_vh) d][4]; a, b: [T][n_vh];
    A_log, dt_bias: [n_vh]; hist_in / hist_out: [3][(2 n_kh + n_vh) d] or None.
    ``out`` may hold preallocated q, k, v, g, beta tensors.  Returns the dict.
    """
    T, cw = qkv.shape
    d = cw // (2 * n_kh + n_vh)
    if d * (2 * n_kh + n_vh) != cw:
        raise ValueError("qkv's row length is not (2 n_kh + n_vh) * d")
    _want(qkv, "qkv", (T, cw))
    _want(conv_w, "conv_w", (cw, 4))
    _want(a, "a", (T, n_vh))
    _want(b, "b", (T, n_vh))
    _want(A_log, "A_log", (n_vh,))
    _want(dt_bias, "dt_bias", (n_vh,))
    for name, h in (("hist_in", hist_in), ("hist_out", hist_out)):
        if h is not None:
            _want(h, name, (3, cw))
    shapes = {"q": (T, n_kh, d), "k": (T, n_kh, d), "v": (T, n_vh, d), "g": (T, n_vh), "beta": (T, n_vh)}
    res = dict(out) if out is not None else {}
    for name, shape in shapes.items():
        if name not in res:
            res[name] = torch.empty(shape, dtype=torch.float32, device=qkv.device)
        _want(res[name], name, shape)
    opt = lambda t: None if t is None else _ptr(t)  # noqa: E731
    lib = load_library()
    rc = lib.gdn_prestage(_ptr(qkv), _ptr(conv_w), opt(hist_in), opt(hist_out), _ptr(a), _ptr(b), _ptr(A_log),
                          _ptr(dt_bias), _ptr(res["q"]), _ptr(res["k"]), _ptr(res["v"]), _ptr(res["g"]),
                          _ptr(res["beta"]), T, n_kh, n_vh, d, int(activation), float(eps), _stream_ptr(stream))
    _check(rc)
    return res


def gdn_recurrence_chunked_noalloc(q, k, v, g, beta, state, out, stream=None):
    """The chunked recurrence through the entry point that allocates nothing.

    For callers that cannot allocate device memory from inside a library (their
    own arena owns the GPU's memory, or the path must not synchronise): ``out``
    must be passed in, and the library's scratch is a fixed static device array
    (at most 96 value heads).  Calls that overlap on the GPU share that array and
    race; serialise them.  Same shapes and results as ``gdn_recurrence(...,
    mode="chunked")``.
    """
    T, n_kh, d = q.shape
    n_vh = v.shape[1]
    _want(q, "q", (T, n_kh, d))
    _want(k, "k", (T, n_kh, d))
    _want(v, "v", (T, n_vh, d))
    _want(g, "g", (T, n_vh))
    _want(beta, "beta", (T, n_vh))
    _want(state, "state", (n_vh, d, d))
    _want(out, "out", (T, n_vh, d))
    lib = load_library()
    rc = lib.gdn_recurrence_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                            _ptr(out), T, n_kh, n_vh, d, _stream_ptr(stream))
    _check(rc)
    return out


def gdn_noalloc_setup(n_kh: int = 16, n_vh: int = 48, d: int = 128, stream=None):
    """The non-allocating entry point's set-up on the current device (a call with
    T = 0): the runtime loads its static scratch, status word and kernels now, so
    a caller can do this at start-up, before it reserves its memory arena and
    before any stream capture."""
    nil = ctypes.c_void_p(0)
    lib = load_library()
    _check(lib.gdn_recurrence_chunked_noalloc(nil, nil, nil, nil, nil, nil, nil, 0, int(n_kh), int(n_vh), int(d),
                                              _stream_ptr(stream)))


def gdn_out_norm(out, z, w, eps: float = 1e-6, y=None, stream=None):
    """Gated RMSNorm of ``out`` ([T][n_vh][d] FP32) with gate ``z`` and weight ``w``
    ([d]) to FP16; returns ``y`` ([T][n_vh][d] float16, allocated if None)."""
    T, n_vh, d = out.shape
    _want(out, "out", (T, n_vh, d))
    _want(z, "z", (T, n_vh, d))
    _want(w, "w", (d,))
    if y is None:
        y = torch.empty((T, n_vh, d), dtype=torch.float16, device=out.device)
    _want(y, "y", (T, n_vh, d), dtype=torch.float16)
    lib = load_library()
    rc = lib.gdn_out_norm(_ptr(out), _ptr(z), _ptr(w), float(eps), _ptr(y), T, n_vh, d, _stream_ptr(stream))
    _check(rc)
    return y


def gdn_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load_library().gdn_device_status(_stream_ptr(stream)))


def gdn_release_scratch(device: int = 0):
    _check(load_library().gdn_release_scratch(int(device)))


def gdn_poison_scratch(bits: int = 0x7FC00000, n_vh: int = 48, stream=None):
    """Fill the chunked-mode scratch with a 32-bit pattern (default: quiet NaN)."""
    _check(load_library().gdn_poison_scratch(int(bits) & 0xFFFFFFFF, int(n_vh), _stream_ptr(stream)))


def gdn_chunked_scratch_bytes(n_vh: int = 48) -> int:
    return int(load_library().gdn_chunked_scratch_bytes(int(n_vh)))


def _option_id(option) -> int:
    return _OPTIONS[option] if isinstance(option, str) else int(option)


def gdn_set_option(option, value):
    """Set a process-wide option of the library (``option``: a GDN_OPT_* number or
    its lower-case name without the prefix, e.g. "chunk_products"; for that one
    ``value`` may also be "mma", "fma" or "tc")."""
    if isinstance(value, str):
        value = _PRODUCTS[value]
    _check(load_library().gdn_set_option(_option_id(option), int(value)))


def gdn_get_option(option) -> int:
    v = ctypes.c_int(0)
    _check(load_library().gdn_get_option(_option_id(option), ctypes.byref(v)))
    return int(v.value)


class options:
    """Context manager: set options for the duration of a block, then restore them.

    >>> with gdn.options(chunk_products="fma", chunk_one_launch=0): ...
    """

    def __init__(self, **kw):
        self.kw = kw
        self.saved = {}

    def __enter__(self):
        for name, value in self.kw.items():
            self.saved[name] = gdn_get_option(name)
            gdn_set_option(name, value)
        return self

    def __exit__(self, *exc):
        for name, value in self.saved.items():
            gdn_set_option(name, value)
        return False


def gdn_launch_count() -> int:
    return int(load_library().gdn_launch_count())


def gdn_last_error() -> str:
    return load_library().gdn_last_error().decode(errors="replace")
