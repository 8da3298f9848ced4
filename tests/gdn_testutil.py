"""Helpers shared by the GPU tests: error metrics, FP16 ulp distance, device
transfers.  Nothing here computes the method; expected values come from the
oracle package only."""
from __future__ import annotations

import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")

# max|diff| / max|value| bound for the FP32 output and state (the north-star
# tolerance; the pages measure at most about 1.1e-6 for their kernels)
TOL = 2e-6


def rel_err(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    assert np.all(np.isfinite(a)), "non-finite values in the GPU result"
    return float(np.max(np.abs(a - ref)) / max(float(np.max(np.abs(ref))), 1e-300))


def fp16_order(bits):
    """Map binary16 bit patterns to integers ordered like the values (+0 == -0)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def fp16_ulp_distance(a_bits, b_bits):
    return np.abs(fp16_order(a_bits) - fp16_order(b_bits))


def fp16_ulp_at(bits):
    """Spacing of binary16 numbers at the magnitude of each value (bits)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int32)
    e = (b >> 10) & 0x1F
    return np.where(e == 0, 2.0 ** -24, 2.0 ** (np.maximum(e, 1) - 25))


def half_bits_to_float(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def parity_token_counts():
    with open(os.path.join(GOLDEN, "pr413_parity_token_counts.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    return [int(x) for x in " ".join(rows).split()]


def page_accuracy_table():
    """{T: (seq_out, seq_state, chunked_out, chunked_state, cvs_out, cvs_state)} from the page."""
    out = {}
    with open(os.path.join(GOLDEN, "pr1372_accuracy_vs_fp64.txt")) as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            parts = ln.split()
            out[int(parts[0])] = tuple(None if p == "-" else float(p) for p in parts[1:])
    return out


def to_dev(x: dict, device="cuda"):
    import torch

    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in x.items()}
