"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things other than itself: a hand-derived
worked example, brute-force products of per-token transfer matrices, closed
forms (beta = 0, the small-beta limit, causal linear attention), the
projection identity of the delta rule, invariances of the prologue,
affinity in the initial state, document isolation, and central finite
differences for the backward pass.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import brute
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng(1234)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _tiny(L=5, K=3, V=4, seed=0, beta_scale=1.0):
    r = np.random.default_rng(seed)
    qh = _unit_rows(r.standard_normal((L, K)))
    kh = _unit_rows(r.standard_normal((L, K)))
    v = r.standard_normal((L, V))
    g = -r.uniform(0.0, 2.0, (L, K))
    beta = beta_scale * r.uniform(0.1, 1.0, L)
    S0 = r.standard_normal((K, V))
    return qh, kh, v, g, beta, S0


# ---------------------------------------------------------------- worked example

def test_worked_example_by_hand():
    with open(os.path.join(GOLDEN, "recurrence_2x2_by_hand.json")) as f:
        ex = json.load(f)
    out, ST = oracle.recurrence(ex["q_hat"], ex["k_hat"], ex["v"], np.log(ex["alpha"]), ex["beta"],
                                ex["scale"], np.array(ex["S0"]))
    np.testing.assert_allclose(out, ex["out"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(ST, ex["S_T"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("with_state", [False, True])
def test_recurrence_matches_unrolled_products(seed, with_state):
    qh, kh, v, g, beta, S0 = _tiny(L=6, K=4, V=3, seed=seed)
    S0 = S0 if with_state else None
    out, ST = oracle.recurrence(qh, kh, v, g, beta, 0.7, S0)
    ob, Sb = brute.unrolled(qh, kh, v, g, beta, 0.7, S0)
    np.testing.assert_allclose(out, ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ST, Sb, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out, brute.attention_form(qh, kh, v, g, beta, 0.7, S0), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_beta_zero_is_pure_decay():
    qh, kh, v, g, beta, S0 = _tiny(L=7, K=4, V=5, seed=3)
    out, ST = oracle.recurrence(qh, kh, v, g, np.zeros(7), 0.5, S0)
    G = np.cumsum(g, axis=0)
    np.testing.assert_allclose(ST, np.exp(G[-1])[:, None] * S0, rtol=1e-13, atol=1e-15)
    exp_out = 0.5 * (qh * np.exp(G)) @ S0
    np.testing.assert_allclose(out, exp_out, rtol=1e-13, atol=1e-15)
    out0, ST0 = oracle.recurrence(qh, kh, v, g, np.zeros(7), 0.5, None)
    assert np.all(out0 == 0) and np.all(ST0 == 0)


def test_small_beta_limit_is_decayed_sum():
    """beta = eps: S_t / eps -> sum_{s<=t} Diag(exp(Gamma_t - Gamma_s)) k_s v_s^T, error O(eps)."""
    qh, kh, v, g, _, _ = _tiny(L=6, K=3, V=2, seed=4)
    G = np.cumsum(g, axis=0)
    for eps in (1e-4, 1e-6):
        out, ST = oracle.recurrence(qh, kh, v, g, np.full(6, eps), 1.0, None)
        Sref = sum(np.exp(G[-1] - G[s])[:, None] * np.outer(kh[s], v[s]) for s in range(6))
        err = np.abs(ST / eps - Sref).max()
        assert err < 50 * eps, err
        for t in range(6):
            St = sum(np.exp(G[t] - G[s])[:, None] * np.outer(kh[s], v[s]) for s in range(t + 1))
            assert np.abs(out[t] / eps - St.T @ qh[t]).max() < 50 * eps


def test_alpha_one_small_beta_is_causal_linear_attention():
    qh, kh, v, _, _, _ = _tiny(L=8, K=4, V=3, seed=5)
    eps = 1e-7
    out, _ = oracle.recurrence(qh, kh, v, np.zeros((8, 4)), np.full(8, eps), 0.25, None)
    ref = 0.25 * np.tril(qh @ kh.T) @ v
    np.testing.assert_allclose(out / eps, ref, rtol=0, atol=1e-5)


def test_single_token_textbook_case():
    r = np.random.default_rng(6)
    q, k = _unit_rows(r.standard_normal((1, 5))), _unit_rows(r.standard_normal((1, 5)))
    v = r.standard_normal((1, 3))
    out, ST = oracle.recurrence(q, k, v, np.zeros((1, 5)), np.ones(1), 0.3, None)
    np.testing.assert_allclose(out[0], 0.3 * float(q[0] @ k[0]) * v[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ST, np.outer(k[0], v[0]), rtol=1e-14, atol=1e-15)


def test_projection_identity_repeated_token():
    """alpha = 1, beta = 1, |k| = 1: I - k k^T is a projection, so a repeated token changes nothing."""
    r = np.random.default_rng(7)
    k = _unit_rows(r.standard_normal((1, 4)))
    v = r.standard_normal((1, 3))
    S0 = r.standard_normal((4, 3))
    kk, vv = np.repeat(k, 2, 0), np.repeat(v, 2, 0)
    _, S1 = oracle.recurrence(k, k, v, np.zeros((1, 4)), np.ones(1), 1.0, S0)
    _, S2 = oracle.recurrence(kk, kk, vv, np.zeros((2, 4)), np.ones(2), 1.0, S0)
    np.testing.assert_allclose(S2, S1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S1.T @ k[0], v[0], rtol=0, atol=1e-13)   # the delta rule writes v exactly


# ---------------------------------------------------------------- prologue

def test_gate_limits_and_special_values():
    lb = -5.0
    for a, d in [(0.0, 0.0), (math.log(16), 0.1), (1.3, -0.2)]:
        assert oracle.gate(-d, a, d, lb) == pytest.approx(lb / 2, abs=1e-15)   # sigmoid(0) = 1/2
        assert oracle.gate(-1e30, a, d, lb) == 0.0                           # alpha = 1 exactly
        assert oracle.gate(1e30, a, d, lb) == lb
        for x in rng0.standard_normal(20) * 3:
            gv = oracle.gate(x, a, d, lb)
            assert lb <= gv <= 0          # closed in floating point: sigmoid saturates
            if abs(math.exp(a) * (x + d)) < 30:
                assert lb < gv < 0
    # a_log = 0, dt_bias = 0 reduces to lb * logistic(g_raw): scipy's logistic
    for x in np.linspace(-8, 8, 33):
        assert oracle.gate(x, 0.0, 0.0, -3.0) == pytest.approx(-3.0 * expit(x), rel=1e-14, abs=1e-300)
    # monotone decreasing in g_raw, steeper with larger a_log
    xs = np.linspace(-3, 3, 50)
    vals = [oracle.gate(x, 1.0, 0.0, lb) for x in xs]
    assert np.all(np.diff(vals) < 0)
    assert abs(oracle.gate(0.5, 2.0, 0.0, lb) - lb / 2) > abs(oracle.gate(0.5, 0.0, 0.0, lb) - lb / 2)


def test_softplus_gate_limits_and_special_values():
    """The unbounded gate g = -exp(a_log) * softplus(g_raw + dt_bias)."""
    sp = lambda x, a, d: oracle.gate(x, a, d, -5.0, "softplus")
    for a, d in [(0.0, 0.0), (math.log(16), 0.1), (1.3, -0.2)]:
        assert sp(-d, a, d) == pytest.approx(-math.exp(a) * math.log(2), rel=1e-15)   # softplus(0) = ln 2
        assert sp(-800.0, a, d) == 0.0                                               # alpha = 1 exactly
        assert sp(60.0, a, d) == pytest.approx(-math.exp(a) * (60.0 + d), rel=1e-15)  # linear for large x
        for x in rng0.standard_normal(20) * 3:
            assert sp(x, a, d) < 0
            assert sp(x, a, d) == oracle.gate(x, a, d, -0.1, "softplus")   # lower_bound is not used
    # unbounded below: far past any lower bound
    assert sp(100.0, math.log(16), 0.0) == pytest.approx(-1600.0, rel=1e-12)
    # a_log = 0, dt_bias = 0 reduces to -softplus(g_raw): numpy's log(e^0 + e^x)
    for x in np.linspace(-30, 30, 61):
        assert sp(x, 0.0, 0.0) == pytest.approx(-np.logaddexp(0.0, x), rel=1e-14, abs=1e-300)
    xs = np.linspace(-3, 3, 50)
    assert np.all(np.diff([sp(x, 1.0, 0.0) for x in xs]) < 0)
    with pytest.raises(ValueError):
        oracle.gate(0.0, 0.0, 0.0, -5.0, "relu")


def test_softplus_gate_full_path_equals_recurrence():
    """With gate="softplus" the full path is the bare recurrence on the numpy-computed decay."""
    d, S0 = _full_inputs(seed=4)
    out, fs = oracle.kda_fwd(**d, initial_state=S0, scale=0.5, lower_bound=-5.0, gate="softplus")
    B, T, H, K = d["q"].shape
    for h in range(H):
        qh = d["q"][0, :, h] / np.sqrt((d["q"][0, :, h] ** 2).sum(-1, keepdims=True) + 1e-6)
        kh = d["k"][0, :, h] / np.sqrt((d["k"][0, :, h] ** 2).sum(-1, keepdims=True) + 1e-6)
        g = -np.exp(d["a_log"][h]) * np.logaddexp(0.0, d["g_raw"][0, :, h] + d["dt_bias"][h * K:(h + 1) * K])
        o, S = oracle.recurrence(qh, kh, d["v"][0, :, h], g, expit(d["beta_raw"][0, :, h]), 0.5, S0[0, h])
        np.testing.assert_allclose(out[0, :, h], o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fs[0, h], S, rtol=1e-12, atol=1e-13)
    # and it differs from the lower-bounded gate on the same logits
    out_lb, _ = oracle.kda_fwd(**d, initial_state=S0, scale=0.5, lower_bound=-5.0)
    assert np.abs(out - out_lb).max() > 1e-3


def _full_inputs(B=1, T=20, H=2, K=4, V=3, seed=0, state=True):
    r = np.random.default_rng(seed)
    d = dict(q=r.standard_normal((B, T, H, K)), k=r.standard_normal((B, T, H, K)),
             v=r.standard_normal((B, T, H, V)), g_raw=r.standard_normal((B, T, H, K)),
             beta_raw=r.standard_normal((B, T, H)), a_log=r.uniform(0, math.log(16), H),
             dt_bias=0.1 * r.standard_normal(H * K))
    S0 = 0.3 * r.standard_normal((B, H, K, V)) if state else None
    return d, S0


def test_prologue_invariances():
    """q and k are L2-normalised and beta = sigmoid(beta_raw): positive rescaling of q or k leaves
    the result unchanged; the result is linear in (v, S0); a huge beta logit means beta = 1."""
    d, S0 = _full_inputs()
    kw = dict(scale=0.5, lower_bound=-5.0)
    out, fs = oracle.kda_fwd(**d, initial_state=S0, **kw)
    d2 = dict(d, q=d["q"] * 3.7, k=d["k"] * 2.5)   # eps / |x|^2 stays ~1e-7
    out2, fs2 = oracle.kda_fwd(**d2, initial_state=S0, **kw)
    np.testing.assert_allclose(out2, out, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(fs2, fs, rtol=1e-5, atol=1e-6)
    out3, fs3 = oracle.kda_fwd(**dict(d, v=2 * d["v"]), initial_state=2 * S0, **kw)
    np.testing.assert_allclose(out3, 2 * out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fs3, 2 * fs, rtol=1e-12, atol=1e-12)
    # the full path equals the bare recurrence on normalised inputs with sigmoid(beta) and the gate
    B, T, H, K = d["q"].shape
    for h in range(H):
        qh = d["q"][0, :, h] / np.sqrt((d["q"][0, :, h] ** 2).sum(-1, keepdims=True) + 1e-6)
        kh = d["k"][0, :, h] / np.sqrt((d["k"][0, :, h] ** 2).sum(-1, keepdims=True) + 1e-6)
        g = np.array([[oracle.gate(d["g_raw"][0, t, h, c], d["a_log"][h], d["dt_bias"][h * K + c], -5.0)
                       for c in range(K)] for t in range(T)])
        o, S = oracle.recurrence(qh, kh, d["v"][0, :, h], g, expit(d["beta_raw"][0, :, h]), 0.5, S0[0, h])
        np.testing.assert_allclose(out[0, :, h], o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fs[0, h], S, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- state and documents

def test_affine_in_initial_state():
    d, Sa = _full_inputs(seed=2)
    _, Sb = _full_inputs(seed=3)
    kw = dict(scale=0.3, lower_bound=-5.0)
    f = lambda S: oracle.kda_fwd(**d, initial_state=S, **kw)
    oab, sab = f(Sa + Sb)
    ob, sb = f(Sb)
    oa, sa = f(Sa)
    o0, s0 = f(None)
    np.testing.assert_allclose(sab - sb, sa - s0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oab - ob, oa - o0, rtol=0, atol=1e-12)


def test_document_isolation():
    lens = [5, 1, 9, 3, 6]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    d, _ = _full_inputs(B=1, T=T, H=2, seed=8, state=False)
    r = np.random.default_rng(9)
    S0 = r.standard_normal((len(lens), 2, 4, 3))
    kw = dict(scale=0.4, lower_bound=-5.0)
    out, fs = oracle.kda_fwd(**d, cu_seqlens=cu, initial_state=S0, **kw)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        dn = {key: (val[:, sl] if val.ndim >= 3 else val) for key, val in d.items()}
        on, fn = oracle.kda_fwd(**dn, initial_state=S0[n:n + 1], **kw)
        np.testing.assert_allclose(out[:, sl], on, rtol=0, atol=1e-14)
        np.testing.assert_allclose(fs[n], fn[0], rtol=0, atol=1e-14)
    # perturbing document 2 moves only document 2
    d2 = {key: val.copy() for key, val in d.items()}
    d2["v"][:, cu[2]:cu[3]] += 1.0
    out2, fs2 = oracle.kda_fwd(**d2, cu_seqlens=cu, initial_state=S0, **kw)
    changed = np.abs(out2 - out).max(axis=(0, 2, 3)) > 0
    assert np.array_equal(np.nonzero(changed)[0], np.arange(cu[2], cu[3]))
    assert np.array_equal(np.nonzero(np.abs(fs2 - fs).max(axis=(1, 2, 3)) > 0)[0], [2])


def test_empty_segment_passes_state_through():
    cu = np.array([0, 4, 4, 10])
    d, _ = _full_inputs(B=1, T=10, H=1, seed=10, state=False)
    S0 = np.random.default_rng(11).standard_normal((3, 1, 4, 3))
    out, fs = oracle.kda_fwd(**d, cu_seqlens=cu, initial_state=S0, scale=0.5, lower_bound=-5.0)
    np.testing.assert_array_equal(fs[1], S0[1])


# ---------------------------------------------------------------- backward

def _loss(res_out, res_fs, dout, dfs):
    return float(np.sum(res_out * dout) + np.sum(res_fs * dfs))


@pytest.mark.parametrize("gate", ["lower_bounded", "softplus"])
@pytest.mark.parametrize("varlen", [False, True])
def test_backward_matches_central_differences(varlen, gate):
    backward_central_differences(varlen, gate)


def backward_central_differences(varlen, gate="lower_bounded"):
    if varlen:
        lens = [3, 5, 2]
        cu = np.concatenate([[0], np.cumsum(lens)])
        d, _ = _full_inputs(B=1, T=10, H=2, K=3, V=2, seed=12, state=False)
        S0 = 0.5 * np.random.default_rng(13).standard_normal((3, 2, 3, 2))
    else:
        cu = None
        d, S0 = _full_inputs(B=2, T=7, H=2, K=3, V=2, seed=14)
    r = np.random.default_rng(15)
    dout = r.standard_normal(d["v"].shape)
    dfs = r.standard_normal(S0.shape)
    kw = dict(scale=0.6, lower_bound=-4.0, gate=gate, cu_seqlens=cu)
    grads = oracle.kda_bwd(**d, dout=dout, initial_state=S0, dfinal_state=dfs, **kw)

    def L(dd, S):
        o, f = oracle.kda_fwd(**dd, initial_state=S, **kw)
        return _loss(o, f, dout, dfs)

    h = 1e-6
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g_raw", "dg_raw"), ("beta_raw", "dbeta_raw"),
             ("a_log", "da_log"), ("dt_bias", "ddt_bias")]
    for name, gname in names:
        x = d[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            num[idx] = (L(dict(d, **{name: xp}), S0) - L(dict(d, **{name: xm}), S0)) / (2 * h)
        err = np.abs(num - grads[gname]).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (name, err)
    num = np.zeros_like(S0)
    for idx in np.ndindex(*S0.shape):
        Sp, Sm = S0.copy(), S0.copy()
        Sp[idx] += h
        Sm[idx] -= h
        num[idx] = (L(d, Sp) - L(d, Sm)) / (2 * h)
    err = np.abs(num - grads["dinitial_state"]).max() / np.abs(num).max()
    assert err < 1e-6, ("S0", err)


def test_backward_long_segment_crosses_checkpoints():
    """150 tokens cross two 64-token checkpoint blocks of the oracle's reverse sweep."""
    d, S0 = _full_inputs(B=1, T=150, H=1, K=3, V=2, seed=16)
    d["g_raw"] -= 4.0            # mild decay so early tokens still matter at the end
    r = np.random.default_rng(17)
    dout = r.standard_normal(d["v"].shape)
    kw = dict(scale=0.6, lower_bound=-5.0)
    grads = oracle.kda_bwd(**d, dout=dout, initial_state=S0, **kw)
    h = 1e-6
    for name, gname in [("k", "dk"), ("g_raw", "dg_raw"), ("v", "dv")]:
        x = d[name]
        for idx in [(0, 0, 0, 0), (0, 63, 0, 1), (0, 64, 0, 1), (0, 100, 0, 0)]:
            if x.ndim == 4 and idx[3] >= x.shape[3]:
                continue
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fp = np.sum(oracle.kda_fwd(**dict(d, **{name: xp}), initial_state=S0, **kw)[0] * dout)
            fm = np.sum(oracle.kda_fwd(**dict(d, **{name: xm}), initial_state=S0, **kw)[0] * dout)
            assert abs((fp - fm) / (2 * h) - grads[gname][idx]) < 1e-6 * max(1.0, abs(grads[gname][idx]))


# ------------------------------------------------------------------ grouped key heads

def _grouped_inputs(B=1, T=9, H=4, Hk=2, K=3, V=2, seed=0):
    """Value-head inputs of _full_inputs with q, k on Hk key heads."""
    d, S0 = _full_inputs(B=B, T=T, H=H, K=K, V=V, seed=seed)
    r = np.random.default_rng(seed + 100)
    d["q"] = r.standard_normal((B, T, Hk, K))
    d["k"] = r.standard_normal((B, T, Hk, K))
    return d, S0


def test_grouped_heads_equal_repeated_keys():
    """H = 4 value heads on Hk = 2 key heads: value head h reads key head h // 2, so the run equals
    the ungrouped run on q, k repeated per value head, and dq, dk are the group sums of that run's
    dq, dk (the chain rule through the repeat)."""
    d, S0 = _grouped_inputs(seed=21)
    G = 2
    rep = dict(d, q=np.repeat(d["q"], G, axis=2), k=np.repeat(d["k"], G, axis=2))
    kw = dict(scale=0.7, lower_bound=-4.0)
    out, fs = oracle.kda_fwd(**d, initial_state=S0, **kw)
    out_r, fs_r = oracle.kda_fwd(**rep, initial_state=S0, **kw)
    np.testing.assert_array_equal(out, out_r)
    np.testing.assert_array_equal(fs, fs_r)
    r = np.random.default_rng(22)
    dout = r.standard_normal(d["v"].shape)
    dfs = r.standard_normal(S0.shape)
    g = oracle.kda_bwd(**d, dout=dout, initial_state=S0, dfinal_state=dfs, **kw)
    g_r = oracle.kda_bwd(**rep, dout=dout, initial_state=S0, dfinal_state=dfs, **kw)
    B, T, Hk, K = d["q"].shape
    for n in ("dq", "dk"):
        assert g[n].shape == (B, T, Hk, K)
        np.testing.assert_allclose(g[n], g_r[n].reshape(B, T, Hk, G, K).sum(axis=3), rtol=1e-12, atol=1e-14)
    for n in ("dv", "dg_raw", "dbeta_raw", "da_log", "ddt_bias", "dinitial_state"):
        np.testing.assert_array_equal(g[n], g_r[n])


def test_grouped_heads_backward_central_differences():
    d, S0 = _grouped_inputs(B=1, T=6, H=4, Hk=2, K=3, V=2, seed=23)
    r = np.random.default_rng(24)
    dout = r.standard_normal(d["v"].shape)
    kw = dict(scale=0.6, lower_bound=-4.0)
    grads = oracle.kda_bwd(**d, dout=dout, initial_state=S0, **kw)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk")):
        x = d[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fp = np.sum(oracle.kda_fwd(**dict(d, **{name: xp}), initial_state=S0, **kw)[0] * dout)
            fm = np.sum(oracle.kda_fwd(**dict(d, **{name: xm}), initial_state=S0, **kw)[0] * dout)
            num[idx] = (fp - fm) / (2 * h)
        err = np.abs(num - grads[gname]).max() / np.abs(num).max()
        assert err < 1e-6, (name, err)


def test_grouped_heads_reject_uneven_groups():
    d, S0 = _grouped_inputs(H=3, Hk=2)
    with pytest.raises(ValueError):
        oracle.kda_fwd(**d, initial_state=S0, scale=0.5, lower_bound=-5.0)


# ------------------------------------------------------------------ short convolution + SiLU prologue

def _conv_inputs(B=2, T=11, C=5, W=4, seed=0):
    r = np.random.default_rng(seed)
    return r.standard_normal((B, T, C)), r.standard_normal((C, W)), r.standard_normal(C)


@pytest.mark.parametrize("W", [1, 2, 4])
def test_short_conv_matches_numpy_convolve(W):
    """Per row and channel the pre-activation is numpy's full convolution with the reversed taps,
    cut to the row length (causal, zero history), plus the bias; then SiLU = a * sigmoid(a)."""
    x, w, b = _conv_inputs(W=W, seed=40 + W)
    y = oracle.short_conv_fwd(x, w, b)
    B, T, C = x.shape
    for bi in range(B):
        for c in range(C):
            a = np.convolve(x[bi, :, c], w[c][::-1])[:T] + b[c]
            np.testing.assert_allclose(y[bi, :, c], a * expit(a), rtol=1e-13, atol=1e-14)
    y0 = oracle.short_conv_fwd(x, w, None)
    a0 = np.stack([np.stack([np.convolve(x[bi, :, c], w[c][::-1])[:T] for c in range(C)], -1) for bi in range(B)])
    np.testing.assert_allclose(y0, a0 * expit(a0), rtol=1e-13, atol=1e-14)


def test_short_conv_matches_depthwise_conv1d():
    """The pages' own formulation: torch conv1d with groups = channels and kernel_size - 1 zero
    padding, output cut to the input length, then SiLU."""
    torch = pytest.importorskip("torch")
    x, w, b = _conv_inputs(B=2, T=9, C=6, W=4, seed=44)
    y = oracle.short_conv_fwd(x, w, b)
    xt = torch.from_numpy(x).transpose(1, 2)
    out = torch.nn.functional.conv1d(xt, torch.from_numpy(w)[:, None, :], torch.from_numpy(b), padding=3, groups=6)
    ref = torch.nn.functional.silu(out[:, :, :9]).transpose(1, 2).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_short_conv_packed_segments_start_from_zero_history():
    lens = [3, 1, 6]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x, w, b = _conv_inputs(B=1, T=10, C=3, W=4, seed=45)
    y = oracle.short_conv_fwd(x, w, b, cu_seqlens=cu)
    for n in range(3):
        s, e = cu[n], cu[n + 1]
        np.testing.assert_array_equal(y[:, s:e], oracle.short_conv_fwd(x[:, s:e], w, b))


@pytest.mark.parametrize("packed", [False, True])
def test_short_conv_backward_central_differences(packed):
    x, w, b = _conv_inputs(B=1 if packed else 2, T=8, C=3, W=3, seed=46)
    cu = np.array([0, 3, 8], dtype=np.int32) if packed else None
    dy = np.random.default_rng(47).standard_normal(x.shape)
    g = oracle.short_conv_bwd(x, w, b, dy, cu_seqlens=cu)
    L = lambda xx, ww, bb: float(np.sum(oracle.short_conv_fwd(xx, ww, bb, cu_seqlens=cu) * dy))
    h = 1e-6
    for name, arr, gname in (("x", x, "dx"), ("w", w, "dweight"), ("b", b, "dbias")):
        num = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = dict(x=x, w=w, b=b)
            args_m = dict(x=x, w=w, b=b)
            args_p[name], args_m[name] = ap, am
            num[idx] = (L(args_p["x"], args_p["w"], args_p["b"]) - L(args_m["x"], args_m["w"], args_m["b"])) / (2 * h)
        err = np.abs(num - g[gname]).max() / np.abs(num).max()
        assert err < 1e-7, (name, err)


def test_state_summary_composes_across_pieces():
    """[P4] state CP: a shard's effect on the state is affine, S_end = M S_begin + S_loc, with M the
    end state from the identity with v = 0 and S_loc the end state from zero.  Cutting one row into
    three pieces and composing the summaries reproduces the whole row's final state and, run from
    the composed entering states, every piece's output (K = V so that M is the state of a run)."""
    d, S0 = _full_inputs(B=1, T=37, H=2, K=3, V=3, seed=31)
    d["g_raw"] -= 3.0            # long memory, so the entering states matter
    kw = dict(scale=0.8, lower_bound=-5.0)
    out, fs = oracle.kda_fwd(**d, initial_state=S0, **kw)
    cuts = [0, 11, 30, 37]
    piece = lambda dd, a, b: {n: (x[:, a:b] if x.ndim >= 3 else x) for n, x in dd.items()}
    eye = np.broadcast_to(np.eye(3), (1, 2, 3, 3)).copy()
    S = S0
    for a, b in zip(cuts[:-1], cuts[1:]):
        p = piece(d, a, b)
        _, S_loc = oracle.kda_fwd(**p, initial_state=None, **kw)
        _, M = oracle.kda_fwd(**dict(p, v=np.zeros_like(p["v"])), initial_state=eye, **kw)
        o_p, f_p = oracle.kda_fwd(**p, initial_state=S, **kw)
        np.testing.assert_allclose(o_p, out[:, a:b], rtol=1e-10, atol=1e-12)
        S_next = np.einsum("nhkl,nhlv->nhkv", M, S) + S_loc
        np.testing.assert_allclose(S_next, f_p, rtol=1e-10, atol=1e-12)
        S = S_next
    np.testing.assert_allclose(S, fs, rtol=1e-10, atol=1e-12)


def test_heads_and_rows_are_equivariant():
    """Heads and batch rows are independent problems: permuting them (with their a_log, dt_bias rows
    and states) permutes every output and gradient the same way.  Catches head / row index mix-ups in
    the per-head parameters (a_log [H], dt_bias [H*K]) and the [N, H, K, V] states."""
    d, S0 = _full_inputs(B=2, T=9, H=3, K=4, V=2, seed=51)
    r = np.random.default_rng(52)
    dout = r.standard_normal(d["v"].shape)
    dfs = r.standard_normal(S0.shape)
    kw = dict(scale=0.6, lower_bound=-4.0)
    ph, pb = [2, 0, 1], [1, 0]
    K = d["q"].shape[-1]
    perm = {n: d[n][pb][:, :, ph] for n in ("q", "k", "v", "g_raw", "beta_raw")}
    perm["a_log"] = d["a_log"][ph]
    perm["dt_bias"] = d["dt_bias"].reshape(-1, K)[ph].reshape(-1)
    S0p = S0[pb][:, ph]
    out, fs = oracle.kda_fwd(**d, initial_state=S0, **kw)
    out_p, fs_p = oracle.kda_fwd(**perm, initial_state=S0p, **kw)
    np.testing.assert_array_equal(out_p, out[pb][:, :, ph])
    np.testing.assert_array_equal(fs_p, fs[pb][:, ph])
    g = oracle.kda_bwd(**d, dout=dout, initial_state=S0, dfinal_state=dfs, **kw)
    g_p = oracle.kda_bwd(**perm, dout=dout[pb][:, :, ph], initial_state=S0p, dfinal_state=dfs[pb][:, ph], **kw)
    for n in ("dq", "dk", "dv", "dg_raw", "dbeta_raw"):
        np.testing.assert_array_equal(g_p[n], g[n][pb][:, :, ph])
    np.testing.assert_allclose(g_p["da_log"], g["da_log"][ph], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g_p["ddt_bias"], g["ddt_bias"].reshape(-1, K)[ph].reshape(-1), rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(g_p["dinitial_state"], g["dinitial_state"][pb][:, ph])


# ------------------------------------------------------------------ gated output norm

def _gn_case(rows=7, V=16, seed=60):
    r = np.random.default_rng(seed)
    return r.standard_normal((rows, V)), r.standard_normal((rows, V)), r.uniform(0.5, 1.5, V)


def test_gated_norm_ungated_limit_is_torch_rms_norm():
    """With the gate saturated (sigmoid = 1) the epilogue is an RMS norm with a weight: torch's
    rms_norm in float64 on the CPU."""
    torch = pytest.importorskip("torch")
    o, _, w = _gn_case()
    y = oracle.gated_norm_fwd(o, np.full_like(o, 800.0), w, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (o.shape[-1],), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)


def test_gated_norm_gate_and_scale():
    """The gate multiplies each element by sigmoid(gate) exactly; with eps = 0 a positive rescaling of a
    row leaves it unchanged; every normalised row has mean square 1 before weight and gate."""
    o, g, w = _gn_case(seed=61)
    y = oracle.gated_norm_fwd(o, g, w, 0.0)
    y1 = oracle.gated_norm_fwd(o, np.full_like(o, 800.0), w, 0.0)
    np.testing.assert_allclose(y, y1 * expit(g), rtol=1e-14, atol=0)
    np.testing.assert_allclose(oracle.gated_norm_fwd(3.7 * o, g, w, 0.0), y, rtol=1e-13, atol=1e-15)
    n = oracle.gated_norm_fwd(o, np.full_like(o, 800.0), np.ones_like(w), 0.0)
    np.testing.assert_allclose((n * n).mean(-1), 1.0, rtol=1e-13)


def test_gated_norm_backward_central_differences():
    o, g, w = _gn_case(rows=3, V=8, seed=62)
    dy = np.random.default_rng(63).standard_normal(o.shape)
    grads = oracle.gated_norm_bwd(o, g, w, 1e-3, dy)
    L = lambda oo, gg, ww: np.sum(oracle.gated_norm_fwd(oo, gg, ww, 1e-3) * dy)
    h = 1e-6
    for name, x, key in (("o", o, "do"), ("gate", g, "dgate"), ("weight", w, "dweight")):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = dict(oo=o, gg=g, ww=w)
            args_m = dict(oo=o, gg=g, ww=w)
            k = {"o": "oo", "gate": "gg", "weight": "ww"}[name]
            args_p[k], args_m[k] = xp, xm
            num[idx] = (L(**args_p) - L(**args_m)) / (2 * h)
        err = np.abs(num - grads[key]).max() / np.abs(num).max()
        assert err < 1e-7, (name, err)
