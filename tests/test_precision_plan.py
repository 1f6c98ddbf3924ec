"""The tensor-core forward's operand precisions, emulated in NumPy against the fp64 oracle (CPU only).

The kernels form the chunkwise algebra (see chunk_model.py) with rounded operands:
  * decayed forms Bkk, Aqk: operands k * exp(Gamma - G_i), exp(G_i - Gamma) k, q * exp(Gamma - G_i) rounded
    to tf32 (nearest), fp32 accumulation, one reference G_i per 16-token row block;
  * W = T Kg with T split into bf16 hi + lo and Kg in bf16; U0 = T v with T split and v exact;
  * the chain: [W; Qg] S, Kd^T U and Aqk U with every operand in fp16, the state in fp32.
These tests run that plan on small workload-shaped inputs and check that the output stays well inside
the bf16 bound (max |x - r| - 2^-8 |r| over rms(r) <= 2e-2), under the workloads' gates and under mild
gates (long memory), and that the fp16 chain is the more accurate choice against a bf16 one (the
8-bit significand of bf16 S, W, Qg is what dominates the error of such a chain).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_sm_gb300.inputs import Workload, make_inputs
from kda_cases import ACT, BF16_ROUNDOFF, TOL_BF16, f64


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def _f16(x):
    return np.asarray(x, np.float64).astype(np.float16).astype(np.float64)


def _tf32(x):
    a = np.asarray(x, np.float32).copy()
    b = a.view(np.uint32)
    b[:] = (b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)   # nearest, ties away, on the 13 dropped bits
    return a.astype(np.float64)


def _split_bf16(x):
    hi = _bf16(x)
    return hi + _bf16(np.asarray(x) - hi)


def _forward(qh, kh, v, g, beta, scale, S0, chain_round):
    """One (row, head) through the kernels' chunkwise forward with their operand roundings."""
    L, K = qh.shape
    S = S0.copy()
    out = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, 64):
        sl = slice(c0, min(L, c0 + 64))
        n = sl.stop - sl.start
        q, k, vv, bt = qh[sl], kh[sl], v[sl], beta[sl]
        G = np.cumsum(np.asarray(g[sl], np.float32), axis=0).astype(np.float64)
        Bkk = np.zeros((n, n))
        Aqk = np.zeros((n, n))
        for i0 in range(0, n, 16):
            i1 = min(n, i0 + 16)
            Gi = G[i0 - 1] if i0 > 0 else np.zeros(K)
            right = _tf32(k[:i1] * np.exp(Gi - G[:i1]))
            Bkk[i0:i1, :i1] = _tf32(k[i0:i1] * np.exp(G[i0:i1] - Gi)) @ right.T
            Aqk[i0:i1, :i1] = _tf32(q[i0:i1] * np.exp(G[i0:i1] - Gi)) @ right.T
        Bkk, Aqk = np.tril(Bkk, -1), np.tril(Aqk)
        Tm = np.linalg.inv(np.eye(n) + bt[:, None] * Bkk) * bt[None, :]
        Kg, Qg = k * np.exp(G), q * np.exp(G)
        Kd, gC = k * np.exp(G[-1] - G), np.exp(G[-1])
        W = _split_bf16(Tm) @ _bf16(Kg)
        U0 = _split_bf16(Tm) @ vv
        r = chain_round
        Sr = r(S)
        U = U0 - r(W) @ Sr
        out[sl] = scale * (r(Qg) @ Sr + r(Aqk) @ r(U))
        S = gC[:, None] * S + r(Kd).T @ r(U)
    return out, S


def _plan_error(g_mean, seed, chain_round, T=512, H=2):
    w = Workload("t", B=1, T=T, H=H, K=128, V=128, initial_state=True, g_mean=g_mean, seed=seed)
    x = make_inputs(w)
    q, k, v, gr, br = (f64(x[n]) for n in ("q", "k", "v", "g_raw", "beta_raw"))
    alog, dtb, S0 = f64(x["a_log"]), f64(x["dt_bias"]), f64(x["initial_state"])
    ref, _ = oracle.kda_fwd(*[f64(x[n]) for n in ACT], scale=x["scale"], lower_bound=x["lower_bound"],
                            initial_state=S0)
    out = np.zeros_like(ref)
    for h in range(H):
        qh, kh = q[0, :, h], k[0, :, h]
        qh = qh / np.sqrt((qh ** 2).sum(1, keepdims=True) + 1e-6)
        kh = kh / np.sqrt((kh ** 2).sum(1, keepdims=True) + 1e-6)
        z = np.exp(alog[h]) * (gr[0, :, h] + dtb.reshape(H, 128)[h])
        g = x["lower_bound"] / (1 + np.exp(-z))
        beta = 1 / (1 + np.exp(-br[0, :, h]))
        out[0, :, h], _ = _forward(qh, kh, v[0, :, h], g, beta, x["scale"], S0[0, h], chain_round)
    ob = _bf16(out)      # the kernel stores the output in bf16
    rms = np.sqrt(np.mean(ref ** 2))
    return max(0.0, float(np.max(np.abs(ob - ref) - BF16_ROUNDOFF * np.abs(ref)))) / rms


@pytest.mark.parametrize("g_mean", [0.0, -4.0], ids=["workload_gates", "mild_gates"])
def test_fp16_chain_plan_is_well_inside_the_bound(g_mean):
    e = max(_plan_error(g_mean, seed, _f16) for seed in (5, 6))
    assert e < 0.5 * TOL_BF16, e


def test_fp16_chain_beats_a_bf16_chain_under_mild_gates():
    e16 = max(_plan_error(-4.0, seed, _f16) for seed in (5, 6))
    eb = max(_plan_error(-4.0, seed, _bf16) for seed in (5, 6))
    assert e16 < 0.7 * eb, (e16, eb)
