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
