"""The seeded synthetic input generator: shapes, distributions, determinism."""
import numpy as np

from linear_attention_recurrence_gb300.inputs import make_inputs


def test_shapes_and_dtypes():
    x = make_inputs(37, seed=1)
    assert x["q"].shape == (37, 16, 128) and x["k"].shape == (37, 16, 128)
    assert x["v"].shape == (37, 48, 128) and x["z"].shape == (37, 48, 128)
    assert x["g"].shape == (37, 48) and x["beta"].shape == (37, 48)
    assert x["S0"].shape == (48, 128, 128) and x["w"].shape == (128,)
    for a in x.values():
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]


def test_distributions():
    x = make_inputs(512, seed=0)
    kn = np.linalg.norm(x["k"].astype(np.float64), axis=-1)
    qn = np.linalg.norm(x["q"].astype(np.float64), axis=-1)
    assert np.allclose(kn, 1.0, atol=1e-6)
    assert np.allclose(qn, 1.0 / np.sqrt(128), atol=1e-7)
    assert np.all(x["g"] < 0)
    assert abs(float(x["g"].mean()) + 0.15) < 0.05  # E[-softplus(N(-2,1))] ~ -0.16
    assert np.all((x["beta"] > 0) & (x["beta"] < 1))
    assert abs(float(x["S0"].std()) - 0.01) < 1e-3
    assert abs(float(x["w"].mean()) - 1.0) < 0.05


def test_deterministic_and_seeded():
    a = make_inputs(16, seed=3, layer=2)
    b = make_inputs(16, seed=3, layer=2)
    c = make_inputs(16, seed=3, layer=3)
    for key in a:
        assert np.array_equal(a[key], b[key])
    assert not np.array_equal(a["v"], c["v"])


def test_prefix_property():
    """A draw for T tokens is the first T tokens of a longer draw."""
    a = make_inputs(40, seed=5)
    b = make_inputs(100, seed=5)
    for key in ("q", "k", "v", "g", "beta", "z"):
        assert np.array_equal(a[key], b[key][:40]), key
    assert np.array_equal(a["S0"], b["S0"]) and np.array_equal(a["w"], b["w"])


def test_prestage_inputs_shapes_and_prefix():
    from linear_attention_recurrence_gb300.inputs import make_prestage_inputs

    a = make_prestage_inputs(40, seed=3, n_kh=2, n_vh=6, d=8)
    b = make_prestage_inputs(25, seed=3, n_kh=2, n_vh=6, d=8)
    cw = (2 * 2 + 6) * 8
    assert a["qkv"].shape == (40, cw) and a["conv_w"].shape == (cw, 4) and a["conv_hist"].shape == (3, cw)
    assert a["a"].shape == (40, 6) and a["A_log"].shape == (6,) and a["dt_bias"].shape == (6,)
    assert all(v.dtype == np.float32 for v in a.values())
    for key in ("qkv", "a", "b"):
        assert np.array_equal(a[key][:25], b[key])
    assert np.all(np.abs(a["conv_w"]) <= 0.5)
    A = np.exp(a["A_log"].astype(np.float64))
    assert np.all((A >= 1.0 - 1e-5) & (A <= 16.0 + 1e-4))
    dt = np.logaddexp(0.0, a["dt_bias"].astype(np.float64))  # softplus(dt_bias) = dt
    assert np.all((dt > 0.9e-3) & (dt < 0.11))
