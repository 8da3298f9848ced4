"""The chunked recurrence entry point that allocates nothing
(gdn_recurrence_chunked_noalloc), called through the C ABI and compared with the
allocating entry point (gdn_recurrence in chunked mode) on two calls in a row.

It exists for callers that cannot let a library allocate device memory: a
serving process whose own arena holds all of the GPU's memory (a cudaMalloc from
inside the library would fail or fragment it), or a path that must not take
cudaMalloc's implicit synchronisation.  Its scratch and its status word are
fixed static device arrays.  This file is named so that pytest collects it last.
"""
import ctypes
import os
import subprocess
import sys

import pytest
import torch

from gdn_testutil import ROOT, to_dev
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
    """The allocating entry point with the warp-MMA products, whose kernels the
    non-allocating one runs."""
    T = b - a
    n_kh, n_vh = t["q"].shape[1], t["v"].shape[1]
    with gdn.options(chunk_products="mma"):
        rc = lib.gdn_recurrence(_p(t["q"][a:b]), _p(t["k"][a:b]), _p(t["v"][a:b]), _p(t["g"][a:b]),
                                _p(t["beta"][a:b]), _p(state), _p(out[a:b]), T, n_kh, n_vh, 128, gdn.GDN_CHUNKED,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == gdn.GDN_OK, lib.gdn_last_error().decode()


@pytest.mark.parametrize("n_kh,T1,T2", [(16, 1300, 777), (32, 513, 64)])
def test_noalloc_within_tolerance_of_the_default_form(lib, n_kh, T1, T2):
    """Against the allocating entry point's default (tensor-memory) form, which
    rounds differently: within the 2e-6 bound of each other's scale."""
    from gdn_testutil import TOL
    x = make_inputs(T1 + T2, seed=21, n_kh=n_kh, n_vh=3 * n_kh, norm=False)
    t = to_dev(x)
    shape = (T1 + T2, 3 * n_kh, 128)
    out_d = torch.full(shape, float("nan"), device="cuda")
    out_n = torch.full(shape, float("nan"), device="cuda")
    st_d = t["S0"].clone()
    st_n = t["S0"].clone()
    for a, b in ((0, T1), (T1, T1 + T2)):
        gdn.gdn_recurrence(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], st_d,
                           out=out_d[a:b], mode="chunked")
        _noalloc(lib, t, a, b, st_n, out_n)
        torch.cuda.synchronize()
        scale = float(out_d[a:b].abs().max())
        assert float((out_n[a:b] - out_d[a:b]).abs().max()) <= 2 * TOL * scale
        assert float((st_n - st_d).abs().max()) <= 2 * TOL * float(st_d.abs().max())
    assert gdn.gdn_device_status() == gdn.GDN_OK


@pytest.mark.parametrize("n_kh,T1,T2", [(16, 1300, 777), (32, 513, 64)])
def test_noalloc_matches_allocating_entry_point(lib, n_kh, T1, T2):
    """Same bits as the allocating path.  Both run the same per-chunk kernels; the
    non-allocating one cuts a call into 512-token super-blocks instead of 2048, but
    super-blocks start on 32-token chunk boundaries and the state passes between
    them through state_inout in FP32, so no rounding differs."""
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
        assert torch.equal(out_n[a:b], out_a[a:b])
        assert torch.equal(st_n, st_a)
    assert torch.isfinite(out_n).all()
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_noalloc_rejects_sizes_beyond_its_maximum(lib):
    nil = ctypes.c_void_p(0)
    rc = lib.gdn_recurrence_chunked_noalloc(nil, nil, nil, nil, nil, nil, nil, 4, 33, 99, 128, nil)
    assert rc == gdn.GDN_ERR_UNSUPPORTED
    msg = lib.gdn_last_error().decode()
    assert "maximum of 96 value heads" in msg, msg


CHILD = r"""
import ctypes, sys, torch
sys.path.insert(0, {root!r})
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs
lib = gdn.load_library()
T = 1300
x = make_inputs(T, seed=4, norm=False)
t = {{k: torch.from_numpy(v).cuda() for k, v in x.items()}}
out = torch.empty((T, 48, 128), device="cuda")
st = t["S0"].clone()
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
nil = ctypes.c_void_p(0)
p = lambda a: ctypes.c_void_p(a.data_ptr())
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
# set-up only (T == 0): the runtime loads the static arrays and the kernels now
assert lib.gdn_recurrence_chunked_noalloc(nil, nil, nil, nil, nil, nil, nil, 0, 16, 48, 128, s) == 0
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
n0 = gdn.gdn_launch_count()
for _ in range(2):
    rc = lib.gdn_recurrence_chunked_noalloc(p(t["q"]), p(t["k"]), p(t["v"]), p(t["g"]), p(t["beta"]), p(st), p(out),
                                            T, 16, 48, 128, s)
    assert rc == 0, lib.gdn_last_error()
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
launches = gdn.gdn_launch_count() - n0
status = gdn.gdn_device_status()
free3 = torch.cuda.mem_get_info()[0]
print("SETUP", free0 - free1, "CALLS", free1 - free3, "LAUNCHES", launches, "STATUS", status,
      "FINITE", bool(torch.isfinite(out).all()))
"""


def test_noalloc_allocates_nothing_in_a_fresh_process():
    """In a process where no other entry point of the library has run: after the
    set-up call (T == 0), two calls leave the device's free memory exactly as it
    was (neither the allocating path's scratch nor its status word appears), and
    the status check afterwards allocates nothing either.  The set-up itself is
    where the runtime, loading modules lazily, sets the static arrays and the
    kernels aside (about 13 MB)."""
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], capture_output=True, text=True,
                       timeout=300, env=dict(os.environ))
    assert r.returncode == 0, r.stderr + r.stdout
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("SETUP")][-1]
    f = line.split()
    setup, calls, launches, status, finite = int(f[1]), int(f[3]), int(f[5]), int(f[7]), f[9]
    assert calls == 0, line
    assert setup <= 64 << 20, line
    assert launches == 2 * 2 * 3, line  # 3 super-blocks of 512 tokens, prep + scan each, two calls
    assert status == gdn.GDN_OK and finite == "True", line

