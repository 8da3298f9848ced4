"""Exact linearity of the GPU recurrence in (v, S0).

The recurrence is linear in the values and the initial state jointly: with q, k, g,
beta fixed, out(2^k v, 2^k S0) = 2^k out(v, S0) and likewise for the final state
("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1", section "What it does": every
product of the chunked form is linear in V and S0; the sequential recurrence of
"#413 prefill: DeltaNet recurrence with the three value heads of a key head in one
thread", section "What changes", likewise).  Scaling by a power of two commutes
with every FP32 rounding (and with the TF32 hi / lo split of the tensor-core form)
as long as nothing over- or underflows, so each kernel must reproduce the scaled
result bit for bit.  A kernel that mixed an operand into the wrong product, or
rounded relative to a fixed scale, fails this at once."""
import contextlib
import os

import numpy as np
import pytest
import torch

from gdn_testutil import to_dev
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_recurrence_gb300 import build

    build.build()


@contextlib.contextmanager
def _scan(kind):
    with gdn.options(chunk_products=kind or "mma"):
        yield


def _run(t, v, s0, mode, kind):
    st = s0.clone()
    with _scan(kind):
        out = gdn.gdn_recurrence(t["q"], t["k"], v, t["g"], t["beta"], st, mode=mode)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    return out.cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("mode,kind", [("sequential", None), ("chunked", "tmem"), ("chunked", None),
                                       ("chunked", "fma"), ("chunked", "tc")])
@pytest.mark.parametrize("e", [-20, 12])
def test_power_of_two_scaling_is_exact(mode, kind, e):
    T = 2100  # a full super-block, a second one of 52 tokens, a ragged last chunk
    t = to_dev(make_inputs(T, seed=31, norm=False))
    o1, s1 = _run(t, t["v"], t["S0"], mode, kind)
    f = 2.0 ** e
    o2, s2 = _run(t, t["v"] * f, t["S0"] * f, mode, kind)
    assert np.isfinite(o1).all() and np.isfinite(s1).all()
    assert np.array_equal((o1 * f).view(np.uint32), o2.view(np.uint32))
    assert np.array_equal((s1 * f).view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("mode,kind", [("sequential", None), ("chunked", "tmem"), ("chunked", None),
                                       ("chunked", "fma")])
def test_heads_do_not_mix(mode, kind):
    """Value head h reads only its own v, g, beta and state and key head h % n_kh:
    changing value head 7's inputs, or key head 3's q and k, leaves every other
    head's output and state bit for bit as it was."""
    T = 700
    t = to_dev(make_inputs(T, seed=32, norm=False))
    o1, s1 = _run(t, t["v"], t["S0"], mode, kind)
    # value head 7: its v and initial state
    v2, s02 = t["v"].clone(), t["S0"].clone()
    v2[:, 7] *= -1.5
    s02[7] += 0.25
    o2, s2 = _run(t, v2, s02, mode, kind)
    other = [h for h in range(48) if h != 7]
    assert np.array_equal(o1[:, other].view(np.uint32), o2[:, other].view(np.uint32))
    assert np.array_equal(s1[other].view(np.uint32), s2[other].view(np.uint32))
    assert not np.array_equal(o1[:, 7], o2[:, 7])
    # key head 3: its q and k reach value heads 3, 19 and 35 only
    t3 = dict(t)
    t3["q"], t3["k"] = t["q"].clone(), t["k"].clone()
    t3["q"][:, 3] = t["q"][:, 3].flip(-1)
    t3["k"][:, 3] = t["k"][:, 3].roll(5, dims=-1)
    o3, s3 = _run(t3, t["v"], t["S0"], mode, kind)
    touched = [3, 19, 35]
    other = [h for h in range(48) if h not in touched]
    assert np.array_equal(o1[:, other].view(np.uint32), o3[:, other].view(np.uint32))
    assert np.array_equal(s1[other].view(np.uint32), s3[other].view(np.uint32))
    for h in touched:
        assert not np.array_equal(o1[:, h], o3[:, h])
