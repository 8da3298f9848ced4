"""FP64 CPU oracle for the Gated DeltaNet prefill recurrence (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library under
``linear_attention_recurrence_gb300`` and its Python binding) never imports it,
and it imports nothing from there.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision); this module
compiles it with gcc and wraps it with ctypes.  Sources, by page title:

* "#413 prefill: DeltaNet recurrence with the three value heads of a key head in
  one thread", section "What changes": the per-token recurrence, the key-head
  sharing ``head % 16`` and the FP16 output norm.
* "#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1 - the prompt's recurrence in
  32-token chunks", section "What it does": the chunked WY form.
* "Round 20 Track C Audit: gdn_pre ... gdn_scan_r ...", section 1 "Summary of
  Changes": the pre-stage's 4-tap causal convolution over the packed qkv rows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_default = None


def compile_library(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library with gcc (OpenMP).

    -ffp-contract=off keeps every product and sum a separately rounded double
    operation on both x86-64 and aarch64.
    """
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into libgdn_oracle.so next to it (if stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, _LIB)
    return _LIB


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes wrapper around one compiled copy of gdn_oracle.c."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        f = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.oracle_gdn_recurrence.argtypes = [f, f, f, f, f, f, f, f, i64, i32, i32, i32, i32]
        lib.oracle_gdn_recurrence.restype = i32
        lib.oracle_gdn_chunked.argtypes = [f, f, f, f, f, f, f, f, i64, i32, i32, i32, i32, i32]
        lib.oracle_gdn_chunked.restype = i32
        lib.oracle_gdn_out_norm.argtypes = [f, f, f, ctypes.c_double, f, i64, i32, i32, i32]
        lib.oracle_gdn_out_norm.restype = i32
        lib.oracle_fp16_rne.argtypes = [ctypes.c_double]
        lib.oracle_fp16_rne.restype = ctypes.c_uint16
        lib.oracle_gdn_prestage.argtypes = [f, f, f, f, f, f, f, i32, ctypes.c_double, f, f, f, f, f, f,
                                            i64, i32, i32, i32]
        lib.oracle_gdn_prestage.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        self.lib = lib

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def recurrence(self, q, k, v, g, beta, S0, nthreads: int | None = None):
        """Sequential FP64 recurrence.  Returns (o [T][n_vh][d], S_final [n_vh][d][d]), float64.

        q, k: [T][n_kh][d]; v: [T][n_vh][d]; g, beta: [T][n_vh]; S0: [n_vh][d][d].
        FP32 inputs are taken exactly as the GPU path sees them (converted to double).
        """
        q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
        T, n_kh, d = q.shape
        n_vh = v.shape[1]
        S_in = _f64(S0).copy()
        S_out = np.empty_like(S_in)
        o = np.empty((T, n_vh, d), dtype=np.float64)
        nt = self.max_threads() if nthreads is None else nthreads
        rc = self.lib.oracle_gdn_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            _ptr(S_in), _ptr(S_out), _ptr(o), T, n_kh, n_vh, d, nt)
        if rc != 0:
            raise RuntimeError(f"oracle_gdn_recurrence failed: {rc}")
        return o, S_out

    def chunked(self, q, k, v, g, beta, S0, C: int = 32, nthreads: int | None = None):
        """FP64 chunked WY form (algebra cross-check).  Same returns as recurrence()."""
        q, k, v, g, beta = _f32(q), _f32(k), _f32(v), _f32(g), _f32(beta)
        T, n_kh, d = q.shape
        n_vh = v.shape[1]
        S_in = _f64(S0).copy()
        S_out = np.empty_like(S_in)
        o = np.empty((T, n_vh, d), dtype=np.float64)
        nt = self.max_threads() if nthreads is None else nthreads
        rc = self.lib.oracle_gdn_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         _ptr(S_in), _ptr(S_out), _ptr(o), T, n_kh, n_vh, d, C, nt)
        if rc != 0:
            raise RuntimeError(f"oracle_gdn_chunked failed: {rc}")
        return o, S_out

    def out_norm(self, o, z, w, eps: float = 1e-6, nthreads: int | None = None):
        """Gated RMSNorm of o ([T][n_vh][d], taken as double) to FP16 bits (uint16 array).

        w is [d], shared by all value heads.
        """
        o = _f64(o)
        z = _f32(z)
        w = _f32(w)
        T, n_vh, d = o.shape
        assert w.shape == (d,)
        y = np.empty((T, n_vh, d), dtype=np.uint16)
        nt = self.max_threads() if nthreads is None else nthreads
        rc = self.lib.oracle_gdn_out_norm(_ptr(o), _ptr(z), _ptr(w), float(eps), _ptr(y),
                                          T, n_vh, d, nt)
        if rc != 0:
            raise RuntimeError(f"oracle_gdn_out_norm failed: {rc}")
        return y

    def prestage(self, qkv, conv_w, hist, a, b, A_log, dt_bias, n_kh: int, n_vh: int, act: int = 1,
                 eps: float = 1e-6):
        """FP64 pre-stage.  Returns dict q, k, v, g, beta, hist (all float64).

        qkv: [T][(2 n_kh + n_vh) d]; conv_w: [(2 n_kh + n_vh) d][4]; hist: [3][Cw] or None;
        a, b: [T][n_vh]; A_log, dt_bias: [n_vh].
        """
        qkv, conv_w, a, b = _f32(qkv), _f32(conv_w), _f32(a), _f32(b)
        A_log, dt_bias = _f32(A_log), _f32(dt_bias)
        T, Cw = qkv.shape
        d = Cw // (2 * n_kh + n_vh)
        assert d * (2 * n_kh + n_vh) == Cw and conv_w.shape == (Cw, 4)
        h_in = None if hist is None else _f32(hist)
        out = {"q": np.empty((T, n_kh, d)), "k": np.empty((T, n_kh, d)), "v": np.empty((T, n_vh, d)),
               "g": np.empty((T, n_vh)), "beta": np.empty((T, n_vh)), "hist": np.empty((3, Cw))}
        rc = self.lib.oracle_gdn_prestage(_ptr(qkv), _ptr(conv_w), None if h_in is None else _ptr(h_in),
                                          _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), int(act), float(eps),
                                          _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]), _ptr(out["g"]),
                                          _ptr(out["beta"]), _ptr(out["hist"]), T, n_kh, n_vh, d)
        if rc != 0:
            raise RuntimeError(f"oracle_gdn_prestage failed: {rc}")
        return out

    def fp16_rne(self, x: float) -> int:
        """The oracle's own double -> binary16 rounding (bits)."""
        return int(self.lib.oracle_fp16_rne(float(x)))


def default() -> Oracle:
    """The oracle built from gdn_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            build()
            _default = Oracle(_LIB)
    return _default


def max_threads() -> int:
    return default().max_threads()


def recurrence(*a, **kw):
    return default().recurrence(*a, **kw)


def chunked(*a, **kw):
    return default().chunked(*a, **kw)


def out_norm(*a, **kw):
    return default().out_norm(*a, **kw)


def prestage(*a, **kw):
    return default().prestage(*a, **kw)


def fp16_rne(x: float) -> int:
    return default().fp16_rne(x)
