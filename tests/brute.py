"""Brute-force forms of the KDA recurrence (NumPy, fp64, tiny inputs only).

These restate the per-token recurrence of "[kimi k3] add eager reference
model with FSDP2" (the explicit recurrent reference of chunk_kda) in a
different shape from the oracle's loop, so that the oracle can be checked
against something other than itself:

* ``unrolled``: every state is a product of per-token transfer matrices,
      S_t = Phi(t, 0) S_0 + sum_{s<=t} Phi(t, s) beta_s k_s v_s^T,
      Phi(t, s) = A_t A_{t-1} ... A_{s+1},  A_r = (I - beta_r k_r k_r^T) Diag(alpha_r),
  built as explicit K x K matrices.
* ``attention_form``: the output as a lower-triangular "attention" sum
      o_t = scale * (S_0^T Phi(t,0)^T q_t + sum_{s<=t} (q_t^T Phi(t,s) beta_s k_s) v_s),
  i.e. each output row is a weighted sum of value rows.
"""
from __future__ import annotations

import numpy as np


def transfer(k, g, beta):
    """A_r = (I - beta k k^T) Diag(exp(g)) for one token."""
    K = k.shape[0]
    return (np.eye(K) - beta * np.outer(k, k)) @ np.diag(np.exp(g))


def phi(ks, gs, betas, t, s):
    """Phi(t, s) = A_t ... A_{s+1} (identity when t == s); tokens are 1-based here."""
    K = ks.shape[1]
    M = np.eye(K)
    for r in range(s + 1, t + 1):
        M = transfer(ks[r - 1], gs[r - 1], betas[r - 1]) @ M
    return M


def unrolled(qh, kh, v, g, beta, scale, S0=None):
    L, K = qh.shape
    V = v.shape[1]
    S0 = np.zeros((K, V)) if S0 is None else S0
    out = np.zeros((L, V))
    S = None
    for t in range(1, L + 1):
        S = phi(kh, g, beta, t, 0) @ S0
        for s in range(1, t + 1):
            S = S + phi(kh, g, beta, t, s) @ (beta[s - 1] * np.outer(kh[s - 1], v[s - 1]))
        out[t - 1] = scale * S.T @ qh[t - 1]
    ST = S if S is not None else S0.copy()
    return out, ST


def attention_form(qh, kh, v, g, beta, scale, S0=None):
    L, K = qh.shape
    V = v.shape[1]
    S0 = np.zeros((K, V)) if S0 is None else S0
    out = np.zeros((L, V))
    for t in range(1, L + 1):
        row = S0.T @ (phi(kh, g, beta, t, 0).T @ qh[t - 1])
        for s in range(1, t + 1):
            wts = qh[t - 1] @ phi(kh, g, beta, t, s) @ (beta[s - 1] * kh[s - 1])
            row = row + wts * v[s - 1]
        out[t - 1] = scale * row
    return out
