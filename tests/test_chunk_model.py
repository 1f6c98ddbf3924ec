"""The chunkwise (WY / UT) algebra the kernels implement equals the oracle's token loop (no GPU)."""
from __future__ import annotations

import numpy as np
import pytest

import chunk_model
import oracle


def _case(L, K, V, seed, mild=False):
    r = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    qh, kh = unit(r.standard_normal((L, K))), unit(r.standard_normal((L, K)))
    v = r.standard_normal((L, V))
    g = -r.uniform(0.0, 0.3 if mild else 5.0, (L, K))
    beta = r.uniform(0.0, 1.0, L)
    S0 = r.standard_normal((K, V))
    return qh, kh, v, g, beta, S0


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("L", [1, 63, 64, 150])
def test_chunk_forward_equals_recurrence(C, L):
    qh, kh, v, g, beta, S0 = _case(L, 8, 6, seed=C * 1000 + L, mild=True)
    o_ref, S_ref = oracle.recurrence(qh, kh, v, g, beta, 0.3, S0)
    o, S = chunk_model.chunk_forward(qh, kh, v, g, beta, 0.3, S0, C=C)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, S_ref, rtol=1e-10, atol=1e-10)


def test_chunk_forward_strong_decay():
    qh, kh, v, g, beta, S0 = _case(200, 16, 8, seed=3)
    o_ref, S_ref = oracle.recurrence(qh, kh, v, g, beta, 0.25, S0)
    o, S = chunk_model.chunk_forward(qh, kh, v, g, beta, 0.25, S0, C=64)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(S, S_ref, rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("C", [4, 64])
def test_chunk_backward_matches_finite_differences(C):
    L, K, V = 11, 3, 2
    qh, kh, v, g, beta, S0 = _case(L, K, V, seed=7, mild=True)
    r = np.random.default_rng(8)
    dO = r.standard_normal((L, V))
    dST = r.standard_normal((K, V))
    res = chunk_model.chunk_backward(qh, kh, v, g, beta, 0.4, dO, S0, dST, C=C)
    args = dict(qh=qh, kh=kh, v=v, g=g, beta=beta, S0=S0)

    def loss(a):
        o, S = oracle.recurrence(a["qh"], a["kh"], a["v"], a["g"], a["beta"], 0.4, a["S0"])
        return float(np.sum(o * dO) + np.sum(S * dST))

    h = 1e-6
    for name, gname in [("qh", "dqh"), ("kh", "dkh"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                        ("S0", "dS0")]:
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            num[idx] = (loss(dict(args, **{name: xp})) - loss(dict(args, **{name: xm}))) / (2 * h)
        err = np.abs(num - res[gname]).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (name, err)


def _forms_case(g, seed=40):
    r = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    C, K = g.shape
    qh, kh = unit(r.standard_normal((C, K))), unit(r.standard_normal((C, K)))
    with np.errstate(over="ignore", invalid="ignore"):   # exp(Gamma_t - Gamma_s) above the diagonal, unused
        z = chunk_model._chunk_quantities(qh, kh, np.zeros((C, 1)), g, np.ones(C))
    return qh, kh, z["Bkk"], z["Aqk"]


def _close(x, ref):
    assert np.isfinite(x).all()
    assert np.abs(x - ref).max() <= 1e-5 * np.abs(ref).max()


def test_subblock_factorisation_holds_for_lower_bound_5_only():
    """The lower-bounded gate's path: with g in (lb, 0) the diagonal sub-block's left factor is at most
    exp(16 |lb|).  In fp32 that holds for lb = -5 (e^80) and overflows for lb = -6 (e^96) once a
    sub-block decays at the bound, which is why the tensor-core path takes lb >= -5 only."""
    r = np.random.default_rng(41)
    for lb, finite in ((-5.0, True), (-6.0, False)):
        g = lb / (1.0 + np.exp(-r.normal(12.0, 1.0, (64, 32))))     # g within 1e-3 of lb
        qh, kh, B_ref, A_ref = _forms_case(g)
        B, A = chunk_model.decayed_forms_subblocks(qh, kh, g, diagonal="factorised")
        if finite:
            _close(B, B_ref)
            _close(A, A_ref)
        else:
            assert not (np.isfinite(B).all() and np.isfinite(A).all())


def test_unbounded_gate_needs_the_direct_diagonal():
    """The unbounded gate -exp(a) softplus(z) with a = ln 16, z ~ N(4, 1): about -64 per token.  The
    factorised diagonal overflows in fp32; factorising only the off-diagonal sub-blocks (both factors
    <= 1) and forming the diagonal blocks from running products of alpha stays finite and exact."""
    r = np.random.default_rng(42)
    g = -16.0 * np.logaddexp(0.0, r.normal(4.0, 1.0, (64, 32)))
    qh, kh, B_ref, A_ref = _forms_case(g)
    B, A = chunk_model.decayed_forms_subblocks(qh, kh, g, diagonal="factorised")
    assert not (np.isfinite(B).all() and np.isfinite(A).all())
    B, A = chunk_model.decayed_forms_subblocks(qh, kh, g, diagonal="direct")
    _close(B, B_ref)
    _close(A, A_ref)
    # and a typical unbounded gate, z ~ N(0, 1), a ~ U(0, ln 16)
    g = -np.exp(r.uniform(0, np.log(16.0), (1, 32))) * np.logaddexp(0.0, r.normal(0.0, 1.0, (64, 32)))
    qh, kh, B_ref, A_ref = _forms_case(g, seed=43)
    B, A = chunk_model.decayed_forms_subblocks(qh, kh, g, diagonal="direct")
    _close(B, B_ref)
    _close(A, A_ref)
