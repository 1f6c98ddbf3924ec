"""Chunkwise (WY / UT-transform) form of the KDA recurrence, NumPy fp64.

This is the algebra the CUDA kernels implement, written plainly so it can be
checked against the token-by-token oracle (it is a different algorithm for
the same result) and used to inspect kernel intermediates.  It is test code:
the CUDA library does not import it.

Per chunk of C tokens with cumulative log-decay Gamma_t = sum_{r<=t} g_r
(0-based inside the chunk) and entering state S0:

    Bkk[t,s] = sum_c k_tc k_sc exp(Gamma_tc - Gamma_sc)        s <  t
    Aqk[t,s] = sum_c q_tc k_sc exp(Gamma_tc - Gamma_sc)        s <= t
    L        = Diag(beta) strict_tril(Bkk)
    T        = (I + L)^-1 Diag(beta)
    Kg = k * exp(Gamma),  Qg = q * exp(Gamma),  Kd = k * exp(Gamma_last - Gamma)
    W  = T Kg,  U0 = T v,  U = U0 - W S0
    O  = scale (Qg S0 + Aqk U)
    S  = Diag(exp(Gamma_last)) S0 + Kd^T U

The backward pass reverses these equations chunk by chunk (see
``chunk_backward``): a reverse chain carries dS across chunks,
    dU  = scale Aqk^T dO + Kd dS_end
    dS0 = Diag(exp(Gamma_last)) dS_end + scale Qg^T dO - W^T dU,
and every other gradient is local to the chunk given S0 and dS_end.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _chunk_quantities(qh, kh, v, g, beta):
    C = qh.shape[0]
    G = np.cumsum(g, axis=0)
    E = np.exp(G[:, None, :] - G[None, :, :])                 # [t, s, c]
    Bkk = np.einsum("tc,sc,tsc->ts", kh, kh, E)
    Aqk = np.tril(np.einsum("tc,sc,tsc->ts", qh, kh, E))
    Lm = beta[:, None] * np.tril(Bkk, -1)
    N = np.linalg.inv(np.eye(C) + Lm)
    Tm = N * beta[None, :]
    Kg = kh * np.exp(G)
    Qg = qh * np.exp(G)
    Kd = kh * np.exp(G[-1][None, :] - G)
    return dict(G=G, E=E, Bkk=np.tril(Bkk, -1), Aqk=Aqk, L=Lm, N=N, T=Tm, Kg=Kg, Qg=Qg, Kd=Kd,
                W=Tm @ Kg, U0=Tm @ v, gC=np.exp(G[-1]))


def decayed_forms_subblocks(qh, kh, g, *, diagonal="factorised", sub=16, dtype=np.float32):
    """Bkk (strictly lower) and Aqk (lower) of one chunk, formed the way the tensor-core kernels do.

    With Gamma cumulative in ``dtype`` and G_{j+1} its value at the end of column sub-block j,
        exp(Gamma_t - Gamma_s) = exp(Gamma_t - G_{j+1}) * exp(G_{j+1} - Gamma_s)     (s in sub-block j).
    The right factor is <= 1; the left is <= 1 for rows past sub-block j.  Rows inside sub-block j take
    it as exp(Gamma_t - G_j) / exp(G_{j+1} - G_j), which nothing bounds: ``diagonal="factorised"`` keeps
    that (the lower-bounded gate's path), ``diagonal="direct"`` forms the diagonal blocks from running
    products of alpha = exp(g) instead (the unbounded gate's path).
    """
    qh, kh, g = (np.asarray(x, dtype=dtype) for x in (qh, kh, g))
    C, K = qh.shape
    G = np.cumsum(g, axis=0, dtype=dtype)
    Bkk = np.zeros((C, C), dtype)
    Aqk = np.zeros((C, C), dtype)
    with np.errstate(over="ignore", invalid="ignore", under="ignore", divide="ignore"):
        for s0 in range(0, C, sub):
            s1 = min(C, s0 + sub)
            Gj = G[s0 - 1] if s0 > 0 else np.zeros(K, dtype)
            Gj1 = G[s1 - 1]
            R = kh[s0:s1] * np.exp(Gj1[None, :] - G[s0:s1])
            if s1 < C:
                Lt = np.exp(G[s1:] - Gj1[None, :])
                Bkk[s1:, s0:s1] = (kh[s1:] * Lt) @ R.T
                Aqk[s1:, s0:s1] = (qh[s1:] * Lt) @ R.T
            if diagonal == "factorised":
                Ld = np.exp(G[s0:s1] - Gj[None, :]) * (dtype(1) / np.exp(Gj1 - Gj))[None, :]
                Bkk[s0:s1, s0:s1] = (kh[s0:s1] * Ld) @ R.T
                Aqk[s0:s1, s0:s1] = (qh[s0:s1] * Ld) @ R.T
            else:
                alpha = np.exp(g[s0:s1])
                for s in range(s1 - s0):
                    e = np.ones(K, dtype)
                    for t in range(s, s1 - s0):
                        if t > s:
                            e = e * alpha[t]
                        w = kh[s0 + s] * e
                        Bkk[s0 + t, s0 + s] = kh[s0 + t] @ w
                        Aqk[s0 + t, s0 + s] = qh[s0 + t] @ w
    return np.tril(Bkk, -1), np.tril(Aqk)


def chunk_forward(qh, kh, v, g, beta, scale, S0=None, C=64):
    """Forward for one segment and one head with the prologue bypassed."""
    L, K = qh.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    out = np.zeros((L, V))
    for c0 in range(0, L, C):
        sl = slice(c0, min(L, c0 + C))
        z = _chunk_quantities(qh[sl], kh[sl], v[sl], g[sl], beta[sl])
        U = z["U0"] - z["W"] @ S
        out[sl] = scale * (z["Qg"] @ S + z["Aqk"] @ U)
        S = z["gC"][:, None] * S + z["Kd"].T @ U
    return out, S


def chunk_backward(qh, kh, v, g, beta, scale, dO, S0=None, dST=None, C=64):
    """Reverse mode of ``chunk_forward``.

    Returns dict(dqh, dkh, dv, dg, dbeta, dS0) -- gradients with respect to
    the normalised q, k, the log-decay g, beta and the entering state.
    """
    L, K = qh.shape
    V = v.shape[1]
    starts = list(range(0, L, C))
    S = np.zeros((K, V)) if S0 is None else np.array(S0, dtype=np.float64)
    S_in = []
    for c0 in starts:                       # forward chain, keep each chunk's entering state
        sl = slice(c0, min(L, c0 + C))
        z = _chunk_quantities(qh[sl], kh[sl], v[sl], g[sl], beta[sl])
        S_in.append(S.copy())
        U = z["U0"] - z["W"] @ S
        S = z["gC"][:, None] * S + z["Kd"].T @ U
    dS = np.zeros((K, V)) if dST is None else np.array(dST, dtype=np.float64)
    res = dict(dqh=np.zeros_like(qh), dkh=np.zeros_like(kh), dv=np.zeros_like(v), dg=np.zeros_like(g),
               dbeta=np.zeros_like(beta))
    for idx in reversed(range(len(starts))):
        c0 = starts[idx]
        sl = slice(c0, min(L, c0 + C))
        q, k, vv, bt, do = qh[sl], kh[sl], v[sl], beta[sl], dO[sl]
        z = _chunk_quantities(q, k, vv, g[sl], bt)
        S0c, dSC = S_in[idx], dS
        G, E, Tm, N = z["G"], z["E"], z["T"], z["N"]
        Vt = vv - z["Kg"] @ S0c
        U = Tm @ Vt
        dU = scale * z["Aqk"].T @ do + z["Kd"] @ dSC
        dY = Tm.T @ dU
        dvv = dY
        dKg = -dY @ S0c.T
        dT = dU @ Vt.T
        dA = np.tril(scale * do @ U.T)
        dQg = scale * do @ S0c.T
        dKd = U @ dSC.T
        dGC = z["gC"] * np.sum(dSC * S0c, axis=1)
        # T = N Diag(beta), N = (I + L)^-1, L = Diag(beta) Bkk (strict lower)
        dN = dT * bt[None, :]
        dbt = np.sum(N * dT, axis=0)
        dL = np.tril(-N.T @ dN @ N.T, -1)
        dbt = dbt + np.sum(dL * z["Bkk"], axis=1)
        dB = bt[:, None] * dL
        # decayed bilinear forms: P[t,s] = sum_c a_tc b_sc E_tsc
        dq = np.einsum("ts,sc,tsc->tc", dA, k, E)
        dk_left = np.einsum("ts,sc,tsc->tc", dB, k, E)
        dk_right = np.einsum("ts,tc,tsc->sc", dA, q, E) + np.einsum("ts,tc,tsc->sc", dB, k, E)
        dG = q * dq + k * dk_left - k * dk_right
        dk = dk_left + dk_right
        eG = np.exp(G)
        eD = np.exp(G[-1][None, :] - G)
        dq = dq + dQg * eG
        dG = dG + dQg * z["Qg"]
        dk = dk + dKg * eG
        dG = dG + dKg * z["Kg"]
        dk = dk + dKd * eD
        dG = dG - dKd * z["Kd"]
        dGlast = dGC + np.sum(dKd * z["Kd"], axis=0)
        dG[-1] += dGlast
        dgc = np.cumsum(dG[::-1], axis=0)[::-1]
        res["dqh"][sl] = dq
        res["dkh"][sl] = dk
        res["dv"][sl] = dvv
        res["dg"][sl] = dgc
        res["dbeta"][sl] = dbt
        dS = z["gC"][:, None] * dSC + scale * z["Qg"].T @ do - z["W"].T @ dU
    res["dS0"] = dS
    return res
