"""Error paths that need a CUDA context: a failed scratch allocation (simulated
on the host) returns GDN_ERR_ALLOC and launches nothing; argument errors from
the binding; no status left behind by normal runs."""
import os
import subprocess
import sys

import pytest
import torch

from gdn_testutil import ROOT, to_dev
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r})
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs
x = make_inputs(64, seed=0, norm=False)
t = {{k: torch.from_numpy(v).cuda() for k, v in x.items()}}
st = t["S0"].clone()
gdn.gdn_set_option("test_fail_scratch_alloc", 1)
n0 = gdn.gdn_launch_count()
try:
    gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st, mode="chunked")
    print("NO-ERROR")
except gdn.GDNError as e:
    torch.cuda.synchronize()
    same = torch.equal(st, t["S0"])
    print("STATUS", e.status, "LAUNCHES", gdn.gdn_launch_count() - n0, "STATE-UNCHANGED", same)
# the sequential mode needs no scratch and still works
gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st, mode="sequential")
torch.cuda.synchronize()
print("SEQ-OK", gdn.gdn_device_status())
"""


def test_simulated_scratch_allocation_failure():
    """In a fresh process (so the scratch has not been allocated yet), the test
    option makes the scratch allocation fail: GDN_ERR_ALLOC, nothing launched."""
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert f"STATUS {gdn.GDN_ERR_ALLOC} LAUNCHES 0 STATE-UNCHANGED True" in r.stdout, r.stdout
    assert "SEQ-OK 0" in r.stdout, r.stdout


def test_binding_rejects_bad_tensors():
    x = make_inputs(8, seed=0, norm=False)
    t = to_dev(x)
    with pytest.raises(ValueError):
        gdn.gdn_recurrence(t["q"].double(), t["k"], t["v"], t["g"], t["beta"], t["S0"].clone())
    with pytest.raises(ValueError):
        gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"][:, :47].contiguous(), t["S0"].clone())
    with pytest.raises(ValueError):
        gdn.gdn_recurrence(t["q"].cpu(), t["k"], t["v"], t["g"], t["beta"], t["S0"].clone())
    with pytest.raises(ValueError):
        gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), mode="fast")
    with pytest.raises(gdn.GDNError) as e:
        # out aliasing v is rejected by the library
        gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), out=t["v"])
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_launch_counter_counts_kernels():
    x = make_inputs(4100, seed=0, norm=False)
    t = to_dev(x)
    n0 = gdn.gdn_launch_count()
    gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), mode="sequential")
    assert gdn.gdn_launch_count() - n0 == 1
    n0 = gdn.gdn_launch_count()
    gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), mode="chunked")
    # per 2048-token super-block: prep and scan in one launch when 8 n_kh scan CTAs
    # leave at least n_kh SMs for the prep, else a prep launch and a scan launch
    one_launch = torch.cuda.get_device_properties(0).multi_processor_count >= 9 * 16
    assert gdn.gdn_launch_count() - n0 == (1 if one_launch else 2) * 3
    torch.cuda.synchronize()


@pytest.mark.parametrize("T", [64, 1000])
def test_bounded_flag_wait_runs_out_and_reports(T):
    """A prep flag that nothing sets (the test hook withholds one task's flag): the
    scan CTAs waiting for it give up after their bounded wait, the kernel ends, and
    gdn_device_status() reports GDN_ERR_TIMEOUT naming the flag; the context stays
    usable and the next call is correct.  At 1000 tokens (32 chunks) the prep tasks
    of that key head's later chunks also wait, bounded, for ring slots that the
    stopped scan CTAs never hand back."""
    import time

    import numpy as np

    import oracle
    from gdn_testutil import TOL, rel_err

    if torch.cuda.get_device_properties(0).multi_processor_count < 9 * 16:
        pytest.skip("too few SMs for the one-launch form")
    x = make_inputs(T, seed=31, norm=False)
    t = to_dev(x)
    st = t["S0"].clone()
    with gdn.options(test_withhold_prep_task=5):  # chunk 0, key head 5
        t0 = time.time()
        gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st, mode="chunked")
        rc = gdn.gdn_device_status()
        elapsed = time.time() - t0
    assert rc == gdn.GDN_ERR_TIMEOUT
    msg = gdn.gdn_last_error()
    assert "prep flag 5" in msg, msg
    if T > 8 * 32 and torch.cuda.get_device_properties(0).multi_processor_count >= 48 + 16:
        assert "tile ring" in msg, msg  # the tensor-memory form's prep also gave up on its ring
    assert elapsed < 30.0
    # the context is usable and the next call is right
    st = t["S0"].clone()
    out = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st, mode="chunked")
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    o_ref, s_ref = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"])
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL and rel_err(st.cpu().numpy(), s_ref) <= TOL
