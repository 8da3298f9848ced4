"""Batched decode step (gdn_decode): each sequence's token against the FP64
oracle's recurrence over that sequence, over several consecutive steps, and
against the prefill path on the same tokens."""
import numpy as np
import pytest
import torch

import oracle
from gdn_testutil import TOL, rel_err, to_dev
from linear_attention_recurrence_gb300 import gdn
from linear_attention_recurrence_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_recurrence_gb300 import build

    build.build()
    oracle.build()


def _batch(B, steps, seed, n_kh=16):
    """B sequences, each with its own inputs for `steps` tokens and its own S0."""
    seqs = [make_inputs(steps, seed=seed, layer=b, n_kh=n_kh, n_vh=3 * n_kh, norm=False) for b in range(B)]
    return seqs


@pytest.mark.parametrize("B,steps,n_kh", [(1, 1, 16), (7, 3, 16), (64, 2, 16), (5, 2, 1)])
def test_decode_matches_oracle(B, steps, n_kh):
    seqs = _batch(B, steps, seed=30, n_kh=n_kh)
    n_vh = 3 * n_kh
    states = torch.from_numpy(np.stack([s["S0"] for s in seqs])).cuda()
    refs = [oracle.recurrence(s["q"], s["k"], s["v"], s["g"], s["beta"], s["S0"]) for s in seqs]
    for t in range(steps):
        step = {name: torch.from_numpy(np.stack([s[name][t] for s in seqs])).cuda()
                for name in ("q", "k", "v", "g", "beta")}
        out = torch.full((B, n_vh, 128), float("nan"), device="cuda")
        gdn.gdn_decode(step["q"], step["k"], step["v"], step["g"], step["beta"], states, out=out)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        for b in range(B):
            assert rel_err(o[b], refs[b][0][t]) <= TOL, (b, t)
    st = states.cpu().numpy()
    for b in range(B):
        assert rel_err(st[b], refs[b][1]) <= TOL, b
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_decode_agrees_with_prefill_path():
    """A decode step per token reproduces the sequential prefill of the same tokens
    (to FP32 rounding: the two kernels sum in different orders)."""
    T = 5
    x = make_inputs(T, seed=31, norm=False)
    t = to_dev(x)
    st_p = t["S0"].clone()
    o_p = gdn.gdn_recurrence(t["q"], t["k"], t["v"], t["g"], t["beta"], st_p, mode="sequential")
    st_d = t["S0"].clone()[None].contiguous()
    outs = []
    for i in range(T):
        outs.append(gdn.gdn_decode(t["q"][i:i + 1], t["k"][i:i + 1], t["v"][i:i + 1], t["g"][i:i + 1],
                                   t["beta"][i:i + 1], st_d))
    torch.cuda.synchronize()
    o_d = torch.cat(outs).cpu().numpy()
    assert rel_err(o_d, o_p.cpu().numpy()) <= TOL
    assert rel_err(st_d[0].cpu().numpy(), st_p.cpu().numpy()) <= TOL


def test_decode_edge_cases():
    nil = None
    x = make_inputs(1, seed=32, norm=False)
    t = to_dev(x)
    # batch 0: nothing happens
    st = t["S0"][None].clone()
    out = torch.empty((0, 48, 128), device="cuda")
    gdn.gdn_decode(t["q"][:0], t["k"][:0], t["v"][:0], t["g"][:0], t["beta"][:0], st[:0], out=out)
    # beta = 0, g = 0: the state is unchanged bit for bit, o = S0^T q
    beta0 = torch.zeros_like(t["beta"])
    g0 = torch.zeros_like(t["g"])
    o = gdn.gdn_decode(t["q"], t["k"], t["v"], g0, beta0, st)
    torch.cuda.synchronize()
    assert torch.equal(st[0], t["S0"])
    ref = np.einsum("hij,hi->hj", x["S0"].astype(np.float64), x["q"][0][np.arange(48) % 16].astype(np.float64))
    assert rel_err(o[0].cpu().numpy(), ref) <= TOL
    with pytest.raises(gdn.GDNError):
        gdn.gdn_decode(t["q"], t["k"], t["v"], t["g"], t["beta"], st, out=t["v"])  # out aliases v
