"""Determinism of the GPU path: sequential mode is bit-identical across reruns
and across T splits that resume from the carried state; chunked mode is
bit-identical across reruns with its scratch poisoned with NaN before each run
("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1", section "Measured": the same
bits on reruns, scratch NaN-filled between runs)."""
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


def _run(t, mode, splits):
    T = t["q"].shape[0]
    st = t["S0"].clone()
    out = torch.full((T, 48, 128), float("nan"), device="cuda")
    a = 0
    for n in splits:
        b = a + n
        gdn.gdn_recurrence(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], st,
                           out=out[a:b], mode=mode)
        a = b
    assert a == T
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    return out.cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("T,splits", [
    (1000, [1, 15, 16, 17, 951]),
    (4099, [2048, 2051]),
    (333, [1] * 20 + [313]),
    (8192, [4096, 1, 4095]),
])
def test_sequential_split_bit_identical(T, splits):
    t = to_dev(make_inputs(T, seed=9, norm=False))
    o1, s1 = _run(t, "sequential", [T])
    o2, s2 = _run(t, "sequential", splits)
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def test_sequential_reruns_bit_identical():
    t = to_dev(make_inputs(2500, seed=10, norm=False))
    o0, s0 = _run(t, "sequential", [2500])
    for _ in range(5):
        o, s = _run(t, "sequential", [2500])
        assert np.array_equal(o0.view(np.uint32), o.view(np.uint32))
        assert np.array_equal(s0.view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("T", [130, 2048, 4099, 8192])
def test_chunked_reruns_bit_identical_with_poisoned_scratch(T):
    t = to_dev(make_inputs(T, seed=11, norm=False))
    gdn.gdn_poison_scratch(0x7FC00000)
    o0, s0 = _run(t, "chunked", [T])
    assert np.all(np.isfinite(o0)) and np.all(np.isfinite(s0))
    for i in range(6):
        gdn.gdn_poison_scratch(0x7FC00000 if i % 2 == 0 else 0xFF800000)
        o, s = _run(t, "chunked", [T])
        assert np.array_equal(o0.view(np.uint32), o.view(np.uint32))
        assert np.array_equal(s0.view(np.uint32), s.view(np.uint32))


def test_norm_reruns_bit_identical():
    x = make_inputs(1000, seed=12)
    t = to_dev(x)
    o = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone())
    y0 = gdn.gdn_out_norm(o, t["z"], t["w"]).cpu().numpy().view(np.uint16)
    for _ in range(3):
        y = gdn.gdn_out_norm(o, t["z"], t["w"]).cpu().numpy().view(np.uint16)
        assert np.array_equal(y0, y)


@pytest.mark.parametrize("T", [1, 127, 128, 1000])
def test_auto_mode_is_the_chosen_mode_bit_for_bit(T):
    """GDN_AUTO runs the sequential kernel below the threshold and the chunked
    kernels from it on, with identical bits to calling that mode directly."""
    t = to_dev(make_inputs(T, seed=13, norm=False))
    chosen = "sequential" if T < gdn.GDN_AUTO_CHUNKED_MIN_T else "chunked"
    oa, sa = _run(t, "auto", [T])
    oc, sc = _run(t, chosen, [T])
    assert np.array_equal(oa.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(sa.view(np.uint32), sc.view(np.uint32))
