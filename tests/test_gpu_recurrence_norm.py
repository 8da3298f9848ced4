"""gdn_recurrence_norm: the recurrence and the gated RMSNorm of its output in one
call.  Its FP32 output must be the bits gdn_recurrence gives, and its FP16 output
the bits gdn_out_norm gives for that output, whichever way the call runs the norm
(in the output epilogue of the tensor-memory chunked scan or of the sequential
scan, inside the warp-MMA one-launch kernel on the SMs that prepare the chunks,
or as a launch after the recurrence), also when the FP32 output is not stored;
and the FP16 output within 1 ulp of the FP64 norm of the same FP32 output ("#413
prefill: DeltaNet recurrence with the three value heads of a key head in one
thread", section "What changes")."""
import numpy as np
import pytest
import torch

import oracle
from gdn_testutil import fp16_ulp_distance, to_dev
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_recurrence_gb300 import build

    build.build()
    oracle.build()


def _one_launch_available():
    return torch.cuda.get_device_properties(0).multi_processor_count >= 9 * 16


def _bits(t):
    return t.cpu().numpy().view(np.uint16 if t.dtype == torch.float16 else np.uint32)


def _pair(t, T, mode):
    """(out, y, state) from gdn_recurrence_norm and from gdn_recurrence + gdn_out_norm."""
    st1 = t["S0"].clone()
    n0 = gdn.gdn_launch_count()
    out1, y1 = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st1, t["z"], t["w"], 1e-6,
                                       mode=mode)
    launches = gdn.gdn_launch_count() - n0
    st2 = t["S0"].clone()
    out2 = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st2, mode=mode)
    y2 = gdn.gdn_out_norm(out2, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    return (out1, y1, st1), (out2, y2, st2), launches


@pytest.mark.parametrize("mode", ["chunked", "sequential", "auto"])
@pytest.mark.parametrize("T", [1, 33, 130, 2048, 4099])
def test_recurrence_norm_matches_the_two_calls(mode, T):
    t = to_dev(make_inputs(T, seed=21))
    (o1, y1, s1), (o2, y2, s2), launches = _pair(t, T, mode)
    assert np.array_equal(_bits(o1), _bits(o2))
    assert np.array_equal(_bits(s1), _bits(s2))
    assert np.array_equal(_bits(y1), _bits(y2))
    chunked = mode == "chunked" or (mode == "auto" and T >= gdn.GDN_AUTO_CHUNKED_MIN_T)
    if chunked and _one_launch_available():
        # with the FP32 output stored: the recurrence, then the norm, per super-block
        assert launches == 2 * ((T + 2047) // 2048)
    if not chunked:
        assert launches == 2  # the scan, then the norm (the fused form is slower when out is stored)


@pytest.mark.parametrize("T", [1, 33, 130, 2048, 4099])
def test_norm_inside_the_one_launch_same_bits(T):
    """Option norm_in_launch=1: the prep CTAs norm each (chunk, key head) once its 8
    scan CTAs have published it, inside the one launch; same bits as the two calls."""
    if not _one_launch_available():
        pytest.skip("too few SMs for the one-launch form")
    t = to_dev(make_inputs(T, seed=25))
    # the in-launch norm belongs to the warp-MMA one-launch kernel
    with gdn.options(norm_in_launch=1, chunk_products="mma"):
        (o1, y1, s1), (o2, y2, s2), launches = _pair(t, T, "chunked")
    assert launches == (T + 2047) // 2048
    assert np.array_equal(_bits(o1), _bits(o2)) and np.array_equal(_bits(s1), _bits(s2))
    assert np.array_equal(_bits(y1), _bits(y2))


def test_recurrence_norm_within_one_ulp_of_fp64():
    T = 777
    x = make_inputs(T, seed=22)
    t = to_dev(x)
    st = t["S0"].clone()
    out, y = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    y_ref = oracle.out_norm(out.double().cpu().numpy(), x["z"], x["w"], 1e-6)
    assert int(fp16_ulp_distance(y.cpu().numpy().view(np.uint16), y_ref).max()) <= 1


def test_recurrence_norm_two_launch_form_same_bits():
    """With the one-launch form off, the norm runs after each super-block's scan:
    same bits."""
    T = 4099
    t = to_dev(make_inputs(T, seed=23))
    st = t["S0"].clone()
    with gdn.options(chunk_products="mma"):  # the form that has both a one- and a two-launch kernel
        o1, y1 = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    with gdn.options(chunk_one_launch=0, chunk_products="mma"):
        st2 = t["S0"].clone()
        n0 = gdn.gdn_launch_count()
        o2, y2 = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st2, t["z"], t["w"], 1e-6)
        torch.cuda.synchronize()
        assert gdn.gdn_launch_count() - n0 == 3 * 3  # prep, scan, norm per super-block
    assert np.array_equal(_bits(o1), _bits(o2)) and np.array_equal(_bits(y1), _bits(y2))


@pytest.mark.parametrize("fused", [0, 1])
def test_recurrence_norm_graph_replay_with_poisoned_outputs(fused):
    """Captured once, replayed with out and y poisoned with NaN and the scratch
    poisoned in between: every replay gives the eager bits (the output flags
    carry the launch's generation number, so no replay norms stale rows)."""
    with gdn.options(norm_in_launch=fused):
        _graph_replay_case()


def _graph_replay_case():
    T = 4099
    t = to_dev(make_inputs(T, seed=24))
    st = t["S0"].clone()
    o_ref, y_ref = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    o_ref, y_ref = _bits(o_ref), _bits(y_ref)
    st = t["S0"].clone()
    out = torch.empty((T, 48, 128), device="cuda")
    y = torch.empty((T, 48, 128), device="cuda", dtype=torch.float16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6, out=out, y=y)
    torch.cuda.synchronize()
    for _ in range(3):
        st.copy_(t["S0"])
        out.fill_(float("nan"))
        y.fill_(float("nan"))
        gdn.gdn_poison_scratch(0x7FC00000)
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == gdn.GDN_OK
        assert np.array_equal(_bits(out), o_ref) and np.array_equal(_bits(y), y_ref)


@pytest.mark.parametrize("T,splits", [(1, [1]), (17, [17]), (4099, [4099]), (4099, [1000, 3099]), (2048, [5, 2043])])
def test_sequential_norm_fused_without_fp32_output(T, splits):
    """Sequential mode fuses the norm into the scan (the 8 CTAs of a key head as
    one cluster, one launch per call) and, asked not to, writes no FP32 output:
    y and the state have the bits of gdn_recurrence followed by gdn_out_norm, also
    when the sequence is split over calls."""
    t = to_dev(make_inputs(T, seed=26))
    st = t["S0"].clone()
    y = torch.full((T, 48, 128), float("nan"), device="cuda", dtype=torch.float16)
    a = 0
    n0 = gdn.gdn_launch_count()
    for n in splits:
        b = a + n
        out, _ = gdn.gdn_recurrence_norm(t["q"][a:b], t["k"][a:b], t["v"][a:b], t["g"][a:b], t["beta"][a:b], st,
                                         t["z"][a:b], t["w"], 1e-6, y=y[a:b], mode="sequential", store_out=False)
        assert out is None
        a = b
    assert gdn.gdn_launch_count() - n0 == len(splits)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    st2 = t["S0"].clone()
    out2 = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st2, mode="sequential")
    y2 = gdn.gdn_out_norm(out2, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), _bits(y2))
    assert np.array_equal(_bits(st), _bits(st2))


@pytest.mark.parametrize("n_kh,T", [(1, 50), (5, 777)])
def test_sequential_norm_fused_other_head_counts(n_kh, T):
    """Other key-head counts for the fused form (8 CTAs per key head)."""
    t = to_dev(make_inputs(T, seed=27, n_kh=n_kh, n_vh=3 * n_kh))
    with gdn.options(norm_in_launch=1):
        (o1, y1, s1), (o2, y2, s2), launches = _pair(t, T, "sequential")
    assert launches == 1
    assert np.array_equal(_bits(o1), _bits(o2)) and np.array_equal(_bits(s1), _bits(s2))
    assert np.array_equal(_bits(y1), _bits(y2))


def test_sequential_norm_fused_graph_replay():
    """The fused sequential call captured once and replayed with y and out poisoned:
    every replay gives the eager bits."""
    with gdn.options(norm_in_launch=1):
        _sequential_fused_graph_case()


def _sequential_fused_graph_case():
    T = 1000
    t = to_dev(make_inputs(T, seed=28))
    st = t["S0"].clone()
    o_ref, y_ref = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6,
                                           mode="sequential")
    torch.cuda.synchronize()
    o_ref, y_ref, s_ref = _bits(o_ref), _bits(y_ref), _bits(st)
    st = t["S0"].clone()
    out = torch.empty((T, 48, 128), device="cuda")
    y = torch.empty((T, 48, 128), device="cuda", dtype=torch.float16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6, out=out,
                                    y=y, mode="sequential")
    torch.cuda.synchronize()
    for _ in range(3):
        st.copy_(t["S0"])
        out.fill_(float("nan"))
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == gdn.GDN_OK
        assert np.array_equal(_bits(out), o_ref) and np.array_equal(_bits(y), y_ref)
        assert np.array_equal(_bits(st), s_ref)


def test_chunked_norm_without_fp32_output_needs_the_tensor_memory_launch():
    """With 48 key heads (144 value heads) the tensor-memory launch does not fit the
    SMs, so the chunked call takes a form that norms the stored FP32 rows: without
    out it is refused, with out it gives the two calls' bits."""
    T, n_kh = 70, 48
    t = to_dev(make_inputs(T, seed=30, n_kh=n_kh, n_vh=3 * n_kh))
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), t["z"], t["w"],
                                1e-6, store_out=False, mode="chunked")
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    (o1, y1, s1), (o2, y2, s2), _ = _pair(t, T, "chunked")
    assert np.array_equal(_bits(o1), _bits(o2)) and np.array_equal(_bits(s1), _bits(s2))
    assert np.array_equal(_bits(y1), _bits(y2))


def test_chunked_norm_warp_mma_form_needs_the_fp32_output():
    """The warp-MMA chunked form norms the stored FP32 rows (after the scan, or read
    back inside its launch): out is required there."""
    t = to_dev(make_inputs(40, seed=27))
    with gdn.options(chunk_products="mma"):
        with pytest.raises(gdn.GDNError) as e:
            gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], t["S0"].clone(), t["z"], t["w"],
                                    1e-6, store_out=False, mode="chunked")
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG
    assert gdn.gdn_device_status() == gdn.GDN_OK


@pytest.mark.parametrize("T,splits", [(1, [1]), (40, [40]), (2048, [2048]), (4099, [4099]), (4099, [1000, 3099]),
                                      (2100, [31, 2069])])
def test_chunked_norm_in_the_epilogue_without_fp32_output(T, splits):
    """The tensor-memory form norms in its output epilogue, so the FP32 output is
    optional: without it, y and the state have the bits of gdn_recurrence +
    gdn_out_norm (also over split calls, ragged chunks and super-blocks), one launch
    per super-block."""
    if not _one_launch_available():
        pytest.skip("too few SMs for the one-launch form")
    t = to_dev(make_inputs(T, seed=28))
    st_ref = t["S0"].clone()
    out_ref = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st_ref, mode="chunked")
    y_ref = gdn.gdn_out_norm(out_ref, t["z"], t["w"], 1e-6)
    st = t["S0"].clone()
    y = torch.full((T, 48, 128), float("nan"), device="cuda", dtype=torch.float16)
    n0 = gdn.gdn_launch_count()
    t0 = 0
    for n in splits:
        sl = slice(t0, t0 + n)
        out, _ = gdn.gdn_recurrence_norm(t["q"][sl], t["k"][sl], t["v"][sl], t["g"][sl], t["beta"][sl], st,
                                         t["z"][sl], t["w"], 1e-6, y=y[sl], mode="chunked", store_out=False)
        assert out is None
        t0 += n
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert gdn.gdn_launch_count() - n0 == sum((n + 2047) // 2048 for n in splits)
    if len(splits) == 1:
        assert np.array_equal(_bits(st), _bits(st_ref))
        assert np.array_equal(_bits(y), _bits(y_ref))
    else:
        # a split changes the chunk boundaries, so compare each call's y with the two
        # calls made on the same split
        st2 = t["S0"].clone()
        t0 = 0
        for n in splits:
            sl = slice(t0, t0 + n)
            o2 = gdn.gdn_recurrence(t["q"][sl], t["k"][sl], t["v"][sl], t["g"][sl], t["beta"][sl], st2, mode="chunked")
            assert np.array_equal(_bits(y[sl]), _bits(gdn.gdn_out_norm(o2, t["z"][sl], t["w"], 1e-6)))
            t0 += n
        torch.cuda.synchronize()
        assert np.array_equal(_bits(st), _bits(st2))


def test_chunked_norm_in_the_epilogue_graph_replay_without_fp32_output():
    """Captured once without the FP32 output, replayed with y poisoned and the
    scratch poisoned in between: every replay gives the eager bits."""
    if not _one_launch_available():
        pytest.skip("too few SMs for the one-launch form")
    T = 4099
    t = to_dev(make_inputs(T, seed=29))
    st = t["S0"].clone()
    _, y_ref = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6,
                                       store_out=False)
    torch.cuda.synchronize()
    y_ref, s_ref = _bits(y_ref), _bits(st)
    st = t["S0"].clone()
    y = torch.empty((T, 48, 128), device="cuda", dtype=torch.float16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6, y=y,
                                    store_out=False)
    torch.cuda.synchronize()
    for _ in range(3):
        st.copy_(t["S0"])
        y.fill_(float("nan"))
        gdn.gdn_poison_scratch(0x7FC00000)
        graph.replay()
        torch.cuda.synchronize()
        assert gdn.gdn_device_status() == gdn.GDN_OK
        assert np.array_equal(_bits(y), y_ref) and np.array_equal(_bits(st), s_ref)


@pytest.mark.parametrize("T", [33, 2048, 4099])
def test_chunked_norm_inside_the_launch_within_one_ulp_of_fp64(T):
    """The tensor-memory form norms in its output epilogue (asked for here with the
    FP32 output stored): one launch per super-block, y within 1 ulp of the FP64 norm
    of the same FP32 output."""
    if not _one_launch_available():
        pytest.skip("too few SMs for the one-launch form")
    x = make_inputs(T, seed=26)
    t = to_dev(x)
    st = t["S0"].clone()
    n0 = gdn.gdn_launch_count()
    with gdn.options(norm_in_launch=1):
        out, y = gdn.gdn_recurrence_norm(t["q"], t["k"], t["v"], t["g"], t["beta"], st, t["z"], t["w"], 1e-6)
    torch.cuda.synchronize()
    assert gdn.gdn_launch_count() - n0 == (T + 2047) // 2048
    assert gdn.gdn_device_status() == gdn.GDN_OK
    y_iso = oracle.out_norm(out.double().cpu().numpy(), x["z"], x["w"], 1e-6)
    assert int(fp16_ulp_distance(_bits(y), y_iso).max()) <= 1
