"""The chunked recurrence entry point that allocates nothing
(gdn_recurrence_chunked_noalloc), called through the C ABI and compared with the
allocating entry point (gdn_recurrence in chunked mode) on two calls in a row.

It exists for callers that cannot let a library allocate device memory (an
arena that owns all of the GPU's memory, or a path that must not synchronise on
cudaMalloc); its scratch is a fixed static device array.  This file is named so
that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gdn_testutil import TOL, rel_err, to_dev
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from linear_attention_recurrence_gb300 import build

    build.build()
    return gdn.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, t, a, b, state, out):
    T = b - a
    n_kh, n_vh = t["q"].shape[1], t["v"].shape[1]
    rc = lib.gdn_recurrence_chunked_noalloc(_p(t["q"][a:b]), _p(t["k"][a:b]), _p(t["v"][a:b]), _p(t["g"][a:b]),
                                            _p(t["beta"][a:b]), _p(state), _p(out[a:b]), T, n_kh, n_vh, 128,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK, lib.gdn_last_error().decode()


def _alloc(lib, t, a, b, state, out):
    T = b - a
    n_kh, n_vh = t["q"].shape[1], t["v"].shape[1]
    rc = lib.gdn_recurrence(_p(t["q"][a:b]), _p(t["k"][a:b]), _p(t["v"][a:b]), _p(t["g"][a:b]),
                            _p(t["beta"][a:b]), _p(state), _p(out[a:b]), T, n_kh, n_vh, 128, gdn.GDN_CHUNKED,
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK, lib.gdn_last_error().decode()


@pytest.mark.parametrize("n_kh,T1,T2", [(16, 1300, 777), (32, 513, 64)])
def test_noalloc_matches_allocating_entry_point(lib, n_kh, T1, T2):
    x = make_inputs(T1 + T2, seed=21, n_kh=n_kh, n_vh=3 * n_kh, norm=False)
    t = to_dev(x)
    shape = (T1 + T2, 3 * n_kh, 128)
    out_a = torch.full(shape, float("nan"), device="cuda")
    out_n = torch.full(shape, float("nan"), device="cuda")
    st_a = t["S0"].clone()
    st_n = t["S0"].clone()
    # two calls in a row, the second continuing from the state the first left
    for a, b in ((0, T1), (T1, T1 + T2)):
        _alloc(lib, t, a, b, st_a, out_a)
        _noalloc(lib, t, a, b, st_n, out_n)
        torch.cuda.synchronize()
        ref_o = out_a[a:b].double().cpu().numpy()
        assert rel_err(out_n[a:b].double().cpu().numpy(), ref_o) <= TOL
        assert rel_err(st_n.double().cpu().numpy(), st_a.double().cpu().numpy()) <= TOL
    assert torch.isfinite(out_n).all()


def test_noalloc_rejects_sizes_beyond_its_maximum(lib):
    nil = ctypes.c_void_p(0)
    rc = lib.gdn_recurrence_chunked_noalloc(nil, nil, nil, nil, nil, nil, nil, 4, 33, 99, 128, nil)
    assert rc == gdn.GDN_ERR_UNSUPPORTED
    msg = lib.gdn_last_error().decode()
    assert "maximum of 96 value heads" in msg, msg
