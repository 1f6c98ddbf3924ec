"""The oracle's pins catch planted mistakes (no GPU).

Each case copies the oracle's C source, plants one plausible mistake (a flipped sign, a dropped
factor, a transposed operand, a wrong index map), compiles the copy and runs the pin battery of
``test_oracle_pins`` against it: at least one pin must fail.  The oracle itself is never modified.
"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

# (what is wrong, exact text in kda_oracle.c, replacement)
MUTATIONS = [
    ("delta-rule write sign", "S[c * V + j] += beta * kh[c] * (v[j] - w[j]);",
     "S[c * V + j] += beta * kh[c] * (v[j] + w[j]);"),
    ("decay exponent sign", "        const double a = exp(g[c]);\n        for (int j = 0; j < V; ++j) S[c * V + j] *= a;",
     "        const double a = exp(-g[c]);\n        for (int j = 0; j < V; ++j) S[c * V + j] *= a;"),
    ("prediction reads q instead of k", "for (int j = 0; j < V; ++j) w[j] += S[c * V + j] * kh[c];",
     "for (int j = 0; j < V; ++j) w[j] += S[c * V + j] * qh[c];"),
    ("output scale applied twice", "o[j] = scale * acc;", "o[j] = scale * scale * acc;"),
    ("L2 norm without the square root", "rq[i] = 1.0 / sqrt(sq + ORACLE_EPS);", "rq[i] = 1.0 / (sq + ORACLE_EPS);"),
    ("gate without the lower bound", "return lower_bound * sigm(z);", "return -sigm(z);"),
    ("decay gradient misses alpha", "dg[i * K + c] += a * acc;", "dg[i * K + c] += acc;"),
    ("beta gradient misses the sigmoid slope", "dbeta_raw[row] = dbeta[i] * beta[i] * (1.0 - beta[i]);",
     "dbeta_raw[row] = dbeta[i] * beta[i];"),
    ("key heads interleaved instead of grouped", "const int hk = h / (H / Hk);", "const int hk = h % Hk;"),
    ("softplus gate sign", "return -exp(a_log) * softplus(g_raw + dt_bias);",
     "return exp(a_log) * softplus(g_raw + dt_bias);"),
    ("softplus gate gradient misses the sigmoid", "const double dx = -dg[i * K + c] * ea * sigm(x);",
     "const double dx = -dg[i * K + c] * ea;"),
    ("dt_bias read channel-major", "oracle_gate_value(g_raw[row * K + c], a_log[h], dt_bias[h * K + c], lb, gate);",
     "oracle_gate_value(g_raw[row * K + c], a_log[h], dt_bias[c * H + h], lb, gate);"),
    ("grouped dq keeps only the last value head", "sq += dqv[vr];", "sq = dqv[vr];"),
    ("SiLU derivative misses the a (1 - s) term", "const double da = dy[t * C + c] * s * (1.0 + a * (1.0 - s));",
     "const double da = dy[t * C + c] * s;"),
    ("convolution gradient crosses document starts", "if (tau < s0) continue;", "if (tau < 0) continue;"),
    ("output gate applied as SiLU", "y[r * V + v] = orow[v] * rn * w[v] * sigm(gate[r * V + v]);",
     "y[r * V + v] = orow[v] * rn * w[v] * gate[r * V + v] * sigm(gate[r * V + v]);"),
    ("norm backward misses the mean term", "d_o[r * V + v] = rn * (dn - n * dot / V);", "d_o[r * V + v] = rn * dn;"),
    ("convolution taps reversed", "if (tau >= s0) a += w[c * W + i] * x[tau * C + c];",
     "if (tau >= s0) a += w[c * W + (W - 1 - i)] * x[tau * C + c];"),
]


def _battery():
    return [
        pins.test_worked_example_by_hand,
        lambda: pins.test_recurrence_matches_unrolled_products(0, True),
        pins.test_beta_zero_is_pure_decay,
        pins.test_small_beta_limit_is_decayed_sum,
        pins.test_alpha_one_small_beta_is_causal_linear_attention,
        pins.test_single_token_textbook_case,
        pins.test_projection_identity_repeated_token,
        pins.test_gate_limits_and_special_values,
        pins.test_prologue_invariances,
        pins.test_affine_in_initial_state,
        pins.test_document_isolation,
        lambda: pins.backward_central_differences(False),
        pins.test_softplus_gate_limits_and_special_values,
        pins.test_softplus_gate_full_path_equals_recurrence,
        lambda: pins.backward_central_differences(False, "softplus"),
        pins.test_heads_and_rows_are_equivariant,
        pins.test_grouped_heads_equal_repeated_keys,
        pins.test_grouped_heads_backward_central_differences,
        lambda: pins.test_short_conv_matches_numpy_convolve(4),
        pins.test_gated_norm_ungated_limit_is_torch_rms_norm,
        pins.test_gated_norm_gate_and_scale,
        pins.test_gated_norm_backward_central_differences,
        lambda: pins.test_short_conv_backward_central_differences(False),
        lambda: pins.test_short_conv_backward_central_differences(True),
    ]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(what, old, new, tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site not found: {what}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", so, str(path), "-lm"], check=True)
    monkeypatch.setattr(oracle, "build", lambda force=False: so)
    monkeypatch.setattr(oracle, "_lib", None)
    failed = []
    for pin in _battery():
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(getattr(pin, "__name__", "pin"))
    assert failed, f"no pin caught the planted mistake: {what}"


def test_unmutated_oracle_passes_the_battery():
    for pin in _battery():
        pin()
    assert os.path.exists(oracle._SRC)
