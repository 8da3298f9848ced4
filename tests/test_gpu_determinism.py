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


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("kind", ["mma", "fma"])
@pytest.mark.parametrize("T", [1, 130, 2048, 4099])
def test_one_launch_chunked_matches_two_launch_bits(T, kind):
    """Prep and scan in one cooperative launch (prep on the SMs the scan leaves
    free, handing records over through flags) give the same bits as the prep
    kernel followed by the scan kernel, with one launch per super-block instead
    of two; for either form of the scan's large products."""
    if _sm_count() < 9 * 16:
        pytest.skip("too few SMs for the one-launch form at 16 key heads")
    t = to_dev(make_inputs(T, seed=14, norm=False))
    n_sb = (T + 2047) // 2048
    with gdn.options(chunk_products=kind):
        with gdn.options(chunk_one_launch=0):
            n0 = gdn.gdn_launch_count()
            o2, s2 = _run(t, "chunked", [T])
            assert gdn.gdn_launch_count() - n0 == 2 * n_sb
        for i in range(3):
            gdn.gdn_poison_scratch(0x7FC00000 if i % 2 == 0 else 0xFF800000)
            n0 = gdn.gdn_launch_count()
            o1, s1 = _run(t, "chunked", [T])
            assert gdn.gdn_launch_count() - n0 == n_sb
            assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
            assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def test_one_launch_chunked_under_graph_replay():
    """A captured chunked call replayed several times, with the scratch poisoned
    with NaN between replays: each replay gives the eager bits.  The flags carry
    a generation number kept in device memory, so a replay cannot take the
    previous replay's flags for its own and read stale (here NaN) records."""
    T = 4099
    t = to_dev(make_inputs(T, seed=15, norm=False))
    o_ref, s_ref = _run(t, "chunked", [T])  # eager; also allocates the scratch before capture
    st = t["S0"].clone()
    out = torch.empty((T, 48, 128), device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st, out=out, mode="chunked")
    torch.cuda.synchronize()
    for i in range(4):
        st.copy_(t["S0"])
        out.fill_(float("nan"))
        gdn.gdn_poison_scratch(0x7FC00000)
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == gdn.GDN_OK
        assert np.array_equal(out.cpu().numpy().view(np.uint32), o_ref.view(np.uint32)), i
        assert np.array_equal(st.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), i


def test_chunked_reruns_at_engine_shapes_with_poisoned_scratch():
    """Chunked mode gives the same bits on 20 reruns at each of seven token counts
    from 130 to 8192, with the scratch filled with NaN (or -inf) before every other
    run ("#1372 DeltaNet recurrence: STRATA_GDN_CHUNKED=1", section "Measured": the
    pages ran 199 reruns at each of 7 engine shapes between 130 and 8192 tokens,
    NaN-filling the scratch between runs)."""
    x = make_inputs(8192, seed=16, norm=False)  # each shape takes a prefix of this draw
    t_all = to_dev(x)
    for T in (130, 257, 1000, 2047, 2049, 4099, 8192):
        t = {k: (v[:T] if k != "S0" else v) for k, v in t_all.items()}
        o_ref, s_ref = _run(t, "chunked", [T])
        for i in range(20):
            if i % 2 == 0:
                gdn.gdn_poison_scratch(0x7FC00000 if i % 4 == 0 else 0xFF800000)
            o, s = _run(t, "chunked", [T])
            assert np.array_equal(o.view(np.uint32), o_ref.view(np.uint32)), (T, i)
            assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), (T, i)


@pytest.mark.parametrize("T", [130, 4099])
def test_tensor_memory_form_same_bits_for_any_prep_cta_count(T):
    """The tensor-memory form's prep CTA count (option chunk_prep_ctas) only changes
    how far the prep runs ahead of the scan: the same bits for 16, 48 and every SM
    the scan leaves, with and without the norm inside the launch."""
    x = make_inputs(T, seed=17)
    t = to_dev(x)
    ref = None
    for n in (0, 16, 48, 4096):
        with gdn.options(chunk_products="tmem", chunk_prep_ctas=n):
            o, s = _run(t, "chunked", [T])
            st = t["S0"].clone()
            out, y = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6)
            torch.cuda.synchronize()
            assert gdn.gdn_device_status() == gdn.GDN_OK
        bits = (o.view(np.uint32), s.view(np.uint32), out.cpu().numpy().view(np.uint32),
                y.cpu().numpy().view(np.uint16))
        if ref is None:
            ref = bits
        else:
            for a, b in zip(ref, bits):
                assert np.array_equal(a, b), n
