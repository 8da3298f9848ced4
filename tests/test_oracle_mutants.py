"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one.  CPU only: each mutant is a textual edit of gdn_oracle.c,
compiled with gcc into a temporary directory; the committed oracle is untouched.
"""
import os

import pytest

import oracle
import oracle_pins

# (name, exact text in gdn_oracle.c, replacement, occurrence to replace (0-based))
MUTANTS = [
    ("drop_decay", "for (size_t e = 0; e < dd; ++e) S[e] *= a;",
     "for (size_t e = 0; e < dd; ++e) S[e] *= 1.0;", 0),
    ("decay_after_kv", "            for (size_t e = 0; e < dd; ++e) S[e] *= a;\n            /* kv = S^T k */",
     "            /* kv = S^T k */", 0),
    ("delta_sign", "delta[j] = b * ((double)vt[j] - kv[j]);",
     "delta[j] = b * ((double)vt[j] + kv[j]);", 0),
    ("drop_beta", "delta[j] = b * ((double)vt[j] - kv[j]);",
     "delta[j] = ((double)vt[j] - kv[j]);", 0),
    ("kv_transposed", "s += S[(size_t)i * d + j] * (double)kt[i];",
     "s += S[(size_t)j * d + i] * (double)kt[i];", 0),
    ("update_transposed", "S[(size_t)i * d + j] += (double)kt[i] * delta[j];",
     "S[(size_t)j * d + i] += (double)kt[i] * delta[j];", 0),
    ("output_uses_k", "s += S[(size_t)i * d + j] * (double)qt[i];",
     "s += S[(size_t)i * d + j] * (double)kt[i];", 0),
    ("key_head_div", "const int kh = h % n_kh;", "const int kh = h / (n_vh / n_kh);", 0),
    ("chunk_gamma_exclusive", "for (int t = 0; t < n; ++t) { run += GATE(t); gam[t] = run; }",
     "for (int t = 0; t < n; ++t) { gam[t] = run; run += GATE(t); }", 0),
    ("chunk_P_no_diagonal", "for (int i = 0; i <= t; ++i) {", "for (int i = 0; i < t; ++i) {", 0),
    ("chunk_A_no_beta", "a = BETA(t) * exp(gam[t] - gam[i]) * kk;", "a = exp(gam[t] - gam[i]) * kk;", 0),
    ("chunk_state_no_decay", "Snew[e] = exp(glast) * S[e];", "Snew[e] = S[e];", 0),
    ("fp16_truncate", "double n = nearbyint(ldexp(ax, 10 - e));", "double n = floor(ldexp(ax, 10 - e));", 0),
    ("norm_sum_not_mean", "sqrt(ss / (double)d + eps)", "sqrt(ss + eps)", 0),
    ("norm_drop_eps", "sqrt(ss / (double)d + eps)", "sqrt(ss / (double)d)", 0),
    ("norm_sigmoid_gate", "const double silu = zj / (1.0 + exp(-zj));",
     "const double silu = 1.0 / (1.0 + exp(-zj));", 0),
    ("norm_drop_weight", "orow[j] * rs * (double)w[j] * silu", "orow[j] * rs * silu", 0),
    ("pre_taps_reversed", "x += (double)conv_w[c * 4 + j] * xr;", "x += (double)conv_w[c * 4 + (3 - j)] * xr;", 0),
    ("pre_drop_history", "xr = hist_in ? (double)hist_in[(3 + r) * Cw + c] : 0.0;", "xr = 0.0;", 0),
    ("pre_history_order", "hist_in[(3 + r) * Cw + c]", "hist_in[(-1 - r) * Cw + c]", 0),
    ("pre_q_no_scale", "sqrt(sq + eps) * sqrt((double)d)", "sqrt(sq + eps)", 0),
    ("pre_k_scaled", "nk = sqrt(sk + eps);", "nk = sqrt(sk + eps) * sqrt((double)d);", 0),
    ("pre_drop_eps", "nk = sqrt(sk + eps);", "nk = sqrt(sk);", 0),
    ("pre_silu_as_sigmoid", "u[c] = act ? x / (1.0 + exp(-x)) : x;", "u[c] = act ? 1.0 / (1.0 + exp(-x)) : x;", 0),
    ("pre_gate_sign", "g[t * n_vh + h] = -exp(", "g[t * n_vh + h] = exp(", 0),
    ("pre_gate_no_exp", "-exp((double)A_log[h])", "-((double)A_log[h])", 0),
    ("pre_gate_drop_bias", "(double)a[t * n_vh + h] + (double)dt_bias[h]", "(double)a[t * n_vh + h]", 0),
    ("pre_beta_tanh", "1.0 / (1.0 + exp(-(double)b[t * n_vh + h]))", "tanh((double)b[t * n_vh + h])", 0),
    ("pre_k_from_q", "const double* uk = u + (int64_t)(n_kh + kh) * d;", "const double* uk = u + (int64_t)kh * d;", 0),
    ("pre_v_offset", "u + (int64_t)(2 * n_kh + h) * d", "u + (int64_t)(n_kh + h) * d", 0),
    ("pre_hist_out_shift", "const int64_t r = T - 3 + i;", "const int64_t r = T - 4 + i;", 0),
    ("pre_softplus_as_exp", "return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));", "return exp(x);", 0),
]


def _mutate(src: str, old: str, new: str, occ: int) -> str:
    pos = -1
    for _ in range(occ + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, occ):
    with open(oracle.SOURCE) as f:
        src = f.read()
    assert old in src, f"mutation site for {name} not found"
    mutant_src = tmp_path / f"{name}.c"
    mutant_src.write_text(_mutate(src, old, new, occ))
    lib = oracle.compile_library(str(mutant_src), str(tmp_path / f"lib{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant {name}"
    os.remove(lib)
