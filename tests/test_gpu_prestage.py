"""GPU parity of the pre-stage ("Round 20 Track C Audit: gdn_pre ...", section 1)
against the FP64 oracle, through the C ABI.

Bar: max|diff| / max|value| <= 2e-6 for q, k, v, g and beta (FP32 outputs of a
4-term convolution, a SiLU, an L2 norm and the gates: a few FP32 roundings each);
the history handed on is a copy, so it must match bit for bit; calls chained
through the history give the bits of one call.
"""
import numpy as np
import pytest
import torch

import oracle
from gdn_testutil import TOL, rel_err
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs, make_prestage_inputs

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_recurrence_gb300 import build

    build.build()
    oracle.build()


def _dev(x):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in x.items()}


def _gpu(t, n_kh, n_vh, hist=True, act=1, hist_out=None, sl=slice(None)):
    res = gdn.gdn_prestage(t["qkv"][sl], t["conv_w"], t["a"][sl], t["b"][sl], t["A_log"], t["dt_bias"], n_kh, n_vh,
                           hist_in=t["conv_hist"] if hist is True else (hist if hist is not False else None),
                           hist_out=hist_out, activation=act)
    torch.cuda.synchronize()
    return {k: res[k].cpu().numpy() for k in KEYS}


def _ref(x, n_kh, n_vh, hist=True, act=1):
    return oracle.prestage(x["qkv"], x["conv_w"], x["conv_hist"] if hist else None, x["a"], x["b"], x["A_log"],
                           x["dt_bias"], n_kh, n_vh, act=act)


def _check(got, ref, where):
    for key in KEYS:
        e = rel_err(got[key], ref[key])
        assert e <= TOL, (where, key, e)


@pytest.mark.parametrize("act", [1, 0])
@pytest.mark.parametrize("hist", [True, False])
def test_prestage_parity_small_T(act, hist):
    """T from 1 (all taps but one on the history) across the 64-token runs."""
    x = make_prestage_inputs(300, seed=1)
    t = _dev(x)
    for T in (1, 2, 3, 4, 5, 63, 64, 65, 130, 300):
        xs = dict(x, qkv=x["qkv"][:T], a=x["a"][:T], b=x["b"][:T])
        ref = _ref(xs, 16, 48, hist=hist, act=act)
        got = _gpu(t, 16, 48, hist=hist, act=act, sl=slice(0, T))
        _check(got, ref, (T, act, hist))


@pytest.mark.parametrize("n_kh,n_vh", [(1, 3), (5, 15), (32, 96), (4, 4)])
def test_prestage_other_head_counts(n_kh, n_vh):
    x = make_prestage_inputs(70, seed=2, n_kh=n_kh, n_vh=n_vh)
    _check(_gpu(_dev(x), n_kh, n_vh), _ref(x, n_kh, n_vh), (n_kh, n_vh))


def test_prestage_history_out_and_chaining():
    """The history handed on is the last three rows (bit for bit, also for T < 3
    where it mixes the incoming history and the new rows); a sequence split into
    calls chained through it gives the bits of one call."""
    T = 200
    x = make_prestage_inputs(T, seed=3)
    t = _dev(x)
    cw = x["qkv"].shape[1]
    full = _gpu(t, 16, 48)
    for n in (0, 1, 2, 3, 5):
        ho = torch.empty((3, cw), device="cuda")
        gdn.gdn_prestage(t["qkv"][:n], t["conv_w"], t["a"][:n], t["b"][:n], t["A_log"], t["dt_bias"], 16, 48,
                         hist_in=t["conv_hist"], hist_out=ho)
        torch.cuda.synchronize()
        want = np.concatenate([x["conv_hist"], x["qkv"][:n]])[-3:]
        assert np.array_equal(ho.cpu().numpy(), want), n
    parts = {k: [] for k in KEYS}
    hist = t["conv_hist"]
    a = 0
    for n in (1, 2, 60, 137):
        ho = torch.empty((3, cw), device="cuda")
        got = _gpu(t, 16, 48, hist=hist, hist_out=ho, sl=slice(a, a + n))
        for k in KEYS:
            parts[k].append(got[k])
        hist = ho
        a += n
    assert a == T
    for k in KEYS:
        assert np.array_equal(np.concatenate(parts[k]).view(np.uint32), full[k].view(np.uint32)), k


def test_prestage_full_size_sampled():
    """The bench's workload (T = 32768, one call): sampled tokens against the
    oracle, each computed from its own four rows."""
    T = 32768
    x = make_prestage_inputs(T, seed=0)
    got = _gpu(_dev(x), 16, 48)
    rng = np.random.default_rng(5)
    sample = sorted(set([0, 1, 2, 3, 63, 64, 65, 1000, T - 1] + list(rng.integers(0, T, 16))))
    col = np.concatenate([x["conv_hist"], x["qkv"]])
    for tk in sample:
        xs = dict(x, qkv=x["qkv"][tk:tk + 1], conv_hist=col[tk:tk + 3], a=x["a"][tk:tk + 1], b=x["b"][tk:tk + 1])
        ref = _ref(xs, 16, 48)
        _check({k: got[k][tk:tk + 1] for k in KEYS}, ref, tk)
    assert all(np.isfinite(got[k]).all() for k in KEYS)


def test_prestage_feeds_the_recurrence():
    """The pre-stage's outputs are valid recurrence inputs: the chunked GPU
    recurrence on them matches the FP64 recurrence of the same FP32 values."""
    T = 300
    x = make_prestage_inputs(T, seed=6)
    t = _dev(x)
    res = gdn.gdn_prestage(t["qkv"], t["conv_w"], t["a"], t["b"], t["A_log"], t["dt_bias"], 16, 48,
                           hist_in=t["conv_hist"])
    S0 = make_inputs(1, seed=6, names=["S0"])["S0"]
    st = torch.from_numpy(S0).cuda()
    out = gdn.gdn_recurrence(res["q"], res["k"], res["v"], res["g"], res["beta"], st, mode="chunked")
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    host = {k: res[k].cpu().numpy() for k in KEYS}
    assert np.all(host["g"] < 0) and np.all((host["beta"] > 0) & (host["beta"] < 1))
    o_ref, s_ref = oracle.recurrence(host["q"], host["k"], host["v"], host["g"], host["beta"], S0)
    assert rel_err(out.cpu().numpy(), o_ref) <= TOL
    assert rel_err(st.cpu().numpy(), s_ref) <= TOL
