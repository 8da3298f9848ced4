"""The C-ABI library loads and exports every function include/gdn.h declares;
host-side argument checks return their status without touching a GPU."""
import ctypes
import os
import re

import pytest

from gdn_testutil import ROOT
from linear_attention_recurrence_gb300 import gdn

HEADER = os.path.join(ROOT, "include", "gdn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from linear_attention_recurrence_gb300 import build, gdn

    build.build()
    return gdn.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "gdn_recurrence" in names and "gdn_out_norm" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_the_header():
    from linear_attention_recurrence_gb300 import gdn

    assert sorted(gdn.EXPORTS) == _declared()


def test_host_side_validation(lib):
    from linear_attention_recurrence_gb300 import gdn

    nil = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)  # never dereferenced: every call below fails its checks first
    r = lib.gdn_recurrence
    assert r(nil, nil, nil, nil, nil, nil, nil, -1, 16, 48, 128, 0, nil) == gdn.GDN_ERR_INVALID_ARG
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 16, 47, 128, 0, nil) == gdn.GDN_ERR_INVALID_ARG
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 16, 48, 128, 7, nil) == gdn.GDN_ERR_INVALID_ARG
    assert r(nil, nil, nil, nil, nil, nil, nil, 0, 16, 48, 128, gdn.GDN_AUTO, nil) == gdn.GDN_OK
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 0, 48, 128, 0, nil) == gdn.GDN_ERR_INVALID_ARG
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 16, 48, 64, 0, nil) == gdn.GDN_ERR_UNSUPPORTED
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 16, 32, 128, 1, nil) == gdn.GDN_ERR_UNSUPPORTED
    assert r(nil, nil, nil, nil, nil, nil, nil, 5, 16, 48, 128, 0, nil) == gdn.GDN_ERR_INVALID_ARG
    assert "null" in lib.gdn_last_error().decode()
    # T == 0 is a no-op, even with null pointers
    assert r(nil, nil, nil, nil, nil, nil, nil, 0, 16, 48, 128, 1, nil) == gdn.GDN_OK
    # misaligned pointers
    bad = ctypes.c_void_p(258)
    assert r(bad, one, one, one, one, one, one, 5, 16, 48, 128, 0, nil) == gdn.GDN_ERR_INVALID_ARG
    n = lib.gdn_out_norm
    assert n(nil, nil, nil, 1e-6, nil, -1, 48, 128, nil) == gdn.GDN_ERR_INVALID_ARG
    assert n(nil, nil, nil, -1.0, nil, 3, 48, 128, nil) == gdn.GDN_ERR_INVALID_ARG
    assert n(nil, nil, nil, float("nan"), nil, 3, 48, 128, nil) == gdn.GDN_ERR_INVALID_ARG
    assert n(nil, nil, nil, 1e-6, nil, 3, 48, 96, nil) == gdn.GDN_ERR_UNSUPPORTED
    assert n(nil, nil, nil, 1e-6, nil, 0, 48, 128, nil) == gdn.GDN_OK
    assert n(nil, nil, nil, 1e-6, nil, 3, 48, 128, nil) == gdn.GDN_ERR_INVALID_ARG


def test_overlap_rejected(lib):
    from linear_attention_recurrence_gb300 import gdn

    base = 1 << 20
    T, nkh, nvh, d = 4, 16, 48, 128
    qk = T * nkh * d * 4
    vb = T * nvh * d * 4
    q = base
    k = q + qk
    v = k + qk
    g = v + vb
    be = g + 4096
    st = be + 4096
    out = v + 256  # inside v
    P = ctypes.c_void_p
    rc = lib.gdn_recurrence(P(q), P(k), P(v), P(g), P(be), P(st), P(out), T, nkh, nvh, d, 0, None)
    assert rc == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()


def test_scratch_size_and_counters(lib):
    # the other forms' records per 2048-token super-block: T'^T, P^T, e^gamma,
    # e^(gamma_last - gamma) per chunk and value head
    records = 64 * 48 * (2 * 32 * 32 + 2 * 32) * 4
    with gdn.options(chunk_products="mma"):
        assert lib.gdn_chunked_scratch_bytes(48) == records
    # the default (tensor-memory) form's tile ring of 8 chunk slots: per slot and key head
    # [K; Q] and K^T as TF32 hi / lo (24576 floats), per slot and value head T', P as hi / lo
    # and the two gate vectors (4160 floats); the scratch holds the larger of the two
    ring = 8 * (16 * 24576 + 48 * 4160) * 4
    assert lib.gdn_chunked_scratch_bytes(48) == max(ring, records)
    assert lib.gdn_chunked_scratch_bytes(0) == 0
    assert lib.gdn_release_scratch(0) == 0
    assert lib.gdn_release_scratch(-1) != 0
    assert lib.gdn_launch_count() >= 0


def test_binding_constants_match_the_header():
    from linear_attention_recurrence_gb300 import gdn

    src = open(HEADER).read()
    assert int(re.search(r"#define GDN_AUTO_CHUNKED_MIN_T (\d+)", src).group(1)) == gdn.GDN_AUTO_CHUNKED_MIN_T
    for name in ("GDN_SEQUENTIAL", "GDN_CHUNKED", "GDN_AUTO", "GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED",
                 "GDN_ERR_ALLOC", "GDN_ERR_CUDA", "GDN_ERR_TIMEOUT"):
        m = re.search(name + r"\s*=\s*(-?\d+)", src)
        assert m and int(m.group(1)) == getattr(gdn, name), name


def test_prestage_host_side_validation(lib):
    from linear_attention_recurrence_gb300 import gdn

    nil = ctypes.c_void_p(0)
    P = ctypes.c_void_p
    f = lib.gdn_prestage

    def call(T=5, n_kh=16, n_vh=48, d=128, act=1, eps=1e-6, ptrs=None):
        ptrs = ptrs if ptrs is not None else [nil] * 13
        return f(*ptrs, T, n_kh, n_vh, d, act, eps, nil)

    assert call(T=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(n_kh=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(act=2) == gdn.GDN_ERR_INVALID_ARG
    assert call(eps=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert call(eps=float("inf")) == gdn.GDN_ERR_INVALID_ARG
    assert call(d=64) == gdn.GDN_ERR_UNSUPPORTED
    assert call() == gdn.GDN_ERR_INVALID_ARG and "null" in lib.gdn_last_error().decode()
    # addresses are never dereferenced: every call below fails its checks first
    T, nkh, nvh, d = 4, 16, 48, 128
    cw = (2 * nkh + nvh) * d
    base = 1 << 24
    qkv = base
    cwt = qkv + T * cw * 4
    a = cwt + cw * 16
    b = a + 4096
    al = b + 4096
    dt = al + 4096
    q = dt + 4096
    k = q + T * nkh * d * 4
    v = k + T * nkh * d * 4
    g = v + T * nvh * d * 4
    be = g + 4096
    good = [P(qkv), P(cwt), nil, nil, P(a), P(b), P(al), P(dt), P(q), P(k), P(v), P(g), P(be)]
    bad = list(good)
    bad[8] = P(q + 4)  # q not 16-byte aligned
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "aligned" in lib.gdn_last_error().decode()
    bad = list(good)
    bad[10] = P(qkv + 256)  # v inside qkv
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()
    bad = list(good)
    bad[11] = P(v + 512)  # g inside v
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()
    bad = list(good)
    bad[2] = P(base + (1 << 26))
    bad[3] = P(base + (1 << 26) + 16)  # history out overlapping history in
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()
    # T == 0 without a history to hand on: a no-op
    zero = [nil, P(cwt), nil, nil, nil, nil, P(al), P(dt), nil, nil, nil, nil, nil]
    assert call(T=0, ptrs=zero) == gdn.GDN_OK


def test_recurrence_norm_host_side_validation(lib):
    from linear_attention_recurrence_gb300 import gdn

    nil = ctypes.c_void_p(0)
    P = ctypes.c_void_p
    f = lib.gdn_recurrence_norm

    def call(T=5, eps=1e-6, ptrs=None, mode=1):
        ptrs = ptrs if ptrs is not None else [nil] * 10
        return f(*ptrs[:9], eps, ptrs[9], T, 16, 48, 128, mode, nil)

    assert call(eps=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert call(eps=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    assert call() == gdn.GDN_ERR_INVALID_ARG and "null" in lib.gdn_last_error().decode()
    assert call(T=0) == gdn.GDN_OK
    T, nkh, nvh, d = 4, 16, 48, 128
    base = 1 << 24
    qk, vb = T * nkh * d * 4, T * nvh * d * 4
    q = base
    k = q + qk
    v = k + qk
    g = v + vb
    be = g + 4096
    st = be + 4096
    out = st + nvh * d * d * 4
    z = out + vb
    w = z + vb
    y = w + 4096
    good = [P(q), P(k), P(v), P(g), P(be), P(st), P(out), P(z), P(w), P(y)]
    bad = list(good)
    bad[9] = P(z + 64)  # y inside z
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()
    bad = list(good)
    bad[9] = P(y + 2)  # y not 8-byte aligned
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "aligned" in lib.gdn_last_error().decode()
    bad = list(good)
    bad[7] = P(out + 256)  # z inside out
    assert call(T=T, ptrs=bad) == gdn.GDN_ERR_INVALID_ARG and "overlap" in lib.gdn_last_error().decode()
