"""Seeded synthetic inputs of the Gated DeltaNet prefill shapes.

This module draws random numbers and shapes them into the distributions below;
it holds none of the recurrence's arithmetic.  Both the CUDA path (through the
tests and the bench) and the FP64 oracle take their inputs from here.

Shapes (all row-major, contiguous, FP32):

* q, k   ``[T][n_kh][d]``: N(0,1), L2-normalised over d per (token, key head)
  in double, q further scaled by 1/sqrt(d), then rounded to FP32.
* v      ``[T][n_vh][d]``: N(0,1).
* g      ``[T][n_vh]``: -softplus(N(-2,1)), always negative (a decay).
* beta   ``[T][n_vh]``: sigmoid(N(0,1)).
* S0     ``[n_vh][d][d]``: N(0, 0.01^2), S0[h][i][j] with i the key dim.
* z      ``[T][n_vh][d]``: N(0,1), the output gate.
* w      ``[d]``: 1 + N(0, 0.1), the norm weight shared by all heads.

Pre-stage inputs (``make_prestage_inputs``), the layer's projections before the
causal convolution:

* qkv     ``[T][(2 n_kh + n_vh) d]``: N(0,1), the packed q, k, v projections.
* conv_w  ``[(2 n_kh + n_vh) d][4]``: U(-0.5, 0.5), the 4 causal taps per channel.
* conv_hist ``[3][(2 n_kh + n_vh) d]``: N(0,1), the three rows before the call.
* a, b    ``[T][n_vh]``: N(0,1), the gate and beta projections.
* A_log   ``[n_vh]``: log U(1, 16); dt_bias ``[n_vh]``: log(e^dt - 1) with
  dt = exp(U(log 1e-3, log 0.1)).

Each tensor comes from its own Philox stream keyed by (seed * 1000 + layer,
tensor id), so tensors can be drawn separately, and a draw for T tokens equals
the first T tokens of a draw for more tokens (the streams are consumed in
row-major order).
"""
from __future__ import annotations

import numpy as np

N_KH = 16
N_VH = 48
D = 128

_IDS = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "S0": 6, "z": 7, "w": 8,
        "qkv": 9, "conv_w": 10, "conv_hist": 11, "a": 12, "b": 13, "A_log": 14, "dt_bias": 15}


def _rng(seed: int, layer: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[seed * 1000 + layer, _IDS[name]]))


def _unit_rows(x: np.ndarray, scale: float) -> np.ndarray:
    n = np.sqrt(np.einsum("...i,...i->...", x, x))[..., None]
    return (x / n * scale).astype(np.float32)


def make_inputs(T: int, seed: int = 0, layer: int = 0, n_kh: int = N_KH, n_vh: int = N_VH,
                d: int = D, norm: bool = True, names=None) -> dict:
    """Draw one layer's inputs for T tokens.

    Returns a dict of numpy arrays with keys q, k, v, g, beta, S0 and, when
    ``norm`` is true, z and w.  ``names`` restricts the draw to a subset.
    """
    want = set(names) if names is not None else set(
        ["q", "k", "v", "g", "beta", "S0"] + (["z", "w"] if norm else []))
    out = {}
    if "q" in want:
        out["q"] = _unit_rows(_rng(seed, layer, "q").standard_normal((T, n_kh, d)), 1.0 / np.sqrt(d))
    if "k" in want:
        out["k"] = _unit_rows(_rng(seed, layer, "k").standard_normal((T, n_kh, d)), 1.0)
    if "v" in want:
        out["v"] = _rng(seed, layer, "v").standard_normal((T, n_vh, d), dtype=np.float32)
    if "g" in want:
        x = _rng(seed, layer, "g").normal(-2.0, 1.0, (T, n_vh))
        out["g"] = (-np.logaddexp(0.0, x)).astype(np.float32)
    if "beta" in want:
        x = _rng(seed, layer, "beta").standard_normal((T, n_vh))
        out["beta"] = (1.0 / (1.0 + np.exp(-x))).astype(np.float32)
    if "S0" in want:
        out["S0"] = (0.01 * _rng(seed, layer, "S0").standard_normal((n_vh, d, d))).astype(np.float32)
    if "z" in want:
        out["z"] = _rng(seed, layer, "z").standard_normal((T, n_vh, d), dtype=np.float32)
    if "w" in want:
        out["w"] = (1.0 + 0.1 * _rng(seed, layer, "w").standard_normal(d)).astype(np.float32)
    return out


def make_prestage_inputs(T: int, seed: int = 0, layer: int = 0, n_kh: int = N_KH, n_vh: int = N_VH,
                         d: int = D) -> dict:
    """Draw one layer's pre-stage inputs for T tokens: qkv, conv_w, conv_hist, a, b,
    A_log, dt_bias (numpy FP32 arrays, shapes in the module docstring)."""
    cw = (2 * n_kh + n_vh) * d
    out = {
        "qkv": _rng(seed, layer, "qkv").standard_normal((T, cw), dtype=np.float32),
        "conv_w": _rng(seed, layer, "conv_w").uniform(-0.5, 0.5, (cw, 4)).astype(np.float32),
        "conv_hist": _rng(seed, layer, "conv_hist").standard_normal((3, cw), dtype=np.float32),
        "a": _rng(seed, layer, "a").standard_normal((T, n_vh), dtype=np.float32),
        "b": _rng(seed, layer, "b").standard_normal((T, n_vh), dtype=np.float32),
        "A_log": np.log(_rng(seed, layer, "A_log").uniform(1.0, 16.0, n_vh)).astype(np.float32),
    }
    dt = np.exp(_rng(seed, layer, "dt_bias").uniform(np.log(1e-3), np.log(0.1), n_vh))
    out["dt_bias"] = np.log(np.expm1(dt)).astype(np.float32)
    return out
