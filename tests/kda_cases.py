"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

ACT = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")

# Tolerances of the quoted workloads: fp32 inputs -> max|x - r| / max|r| <= 1e-4;
# bf16 inputs with fp32 state -> max|x - r| / rms(r) <= 2e-2 (per tensor).
TOL_FP32 = 1e-4
TOL_BF16 = 2e-2


def f64(t):
    if t is None or isinstance(t, np.ndarray):
        return t
    return t.detach().to(torch.float64).cpu().numpy()


# Storing a result in bf16 rounds it by up to half an ulp, i.e. up to 2^-8 of its magnitude; the
# tolerance bounds the computation's error, so that storage rounding is allowed on top of it.
BF16_ROUNDOFF = 2.0 ** -8


def rel_err(x, r, dtype):
    """Normalised max error of ``x`` against the oracle ``r``.

    fp32 workloads: max|x - r| / max|r|.  bf16 workloads: max(|x - r| - u|r|) / rms(r), with
    u = 2^-8 when ``x`` itself is stored in bf16 (its own rounding) and u = 0 for fp32 results.
    """
    u = BF16_ROUNDOFF if isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16 else 0.0
    x = f64(x) if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    d = np.max(np.abs(x - r) - u * np.abs(r)) if r.size else 0.0
    d = max(d, 0.0)
    if dtype == "fp32":
        den = np.abs(r).max() if r.size else 1.0
    else:
        den = np.sqrt(np.mean(r * r)) if r.size else 1.0
    return float(d / max(den, 1e-30))


def tol(dtype):
    return TOL_FP32 if dtype == "fp32" else TOL_BF16


def head_slice(x: dict, heads) -> dict:
    """Restrict every per-head input to the listed heads (for sampled oracle runs)."""
    heads = list(heads)
    assert x["q"].shape[2] == x["v"].shape[2], "head_slice takes ungrouped inputs (one key head per value head)"
    K = x["q"].shape[-1]
    out = dict(x)
    for n in ("q", "k", "v", "g_raw", "dout"):
        if x.get(n) is not None:
            out[n] = x[n][:, :, heads]
    out["beta_raw"] = x["beta_raw"][:, :, heads]
    out["a_log"] = x["a_log"][heads]
    out["dt_bias"] = x["dt_bias"].view(-1, K)[heads].reshape(-1)
    if x.get("initial_state") is not None:
        out["initial_state"] = x["initial_state"][:, heads]
    return out


def oracle_fwd(x: dict, rows=None):
    """Oracle forward on the inputs ``x`` (optionally only batch rows ``rows`` when not packed)."""
    xs = dict(x)
    if rows is not None:
        assert x.get("cu_seqlens") is None
        for n in ("q", "k", "v", "g_raw", "beta_raw", "dout"):
            if xs.get(n) is not None:
                xs[n] = xs[n][rows]
        if xs.get("initial_state") is not None:
            xs["initial_state"] = xs["initial_state"][rows]
    cu = f64(xs["cu_seqlens"]).astype(np.int64) if xs.get("cu_seqlens") is not None else None
    return oracle.kda_fwd(*[f64(xs[n]) for n in ACT], scale=xs["scale"], lower_bound=xs["lower_bound"],
                          gate=xs.get("gate", "lower_bounded"), cu_seqlens=cu, initial_state=f64(xs.get("initial_state")))


def oracle_bwd(x: dict, rows=None, dfinal=None):
    xs = dict(x)
    if rows is not None:
        assert x.get("cu_seqlens") is None
        for n in ("q", "k", "v", "g_raw", "beta_raw", "dout"):
            if xs.get(n) is not None:
                xs[n] = xs[n][rows]
        if xs.get("initial_state") is not None:
            xs["initial_state"] = xs["initial_state"][rows]
        if dfinal is not None:
            dfinal = dfinal[rows]
    cu = f64(xs["cu_seqlens"]).astype(np.int64) if xs.get("cu_seqlens") is not None else None
    return oracle.kda_bwd(*[f64(xs[n]) for n in ACT], f64(xs["dout"]), scale=xs["scale"],
                          lower_bound=xs["lower_bound"], gate=xs.get("gate", "lower_bounded"), cu_seqlens=cu,
                          initial_state=f64(xs.get("initial_state")),
                          dfinal_state=f64(dfinal))


def gpu_fwd(x: dict, simt=False, final=True, segments=0):
    import gated_delta_rule_sm_gb300 as kda
    return kda.forward(*[x[n] for n in ACT], scale=x["scale"], lower_bound=x["lower_bound"],
                       gate=x.get("gate", "lower_bounded"), chunk_size=x.get("chunk_size", 64), cu_seqlens=x.get("cu_seqlens"),
                       initial_state=x.get("initial_state"), output_final_state=final, simt=simt, segments=segments)


def gpu_bwd(x: dict, dfinal=None, segments=0):
    import gated_delta_rule_sm_gb300 as kda
    return kda.backward(*[x[n] for n in ACT], x["dout"], scale=x["scale"], lower_bound=x["lower_bound"],
                        gate=x.get("gate", "lower_bounded"), chunk_size=x.get("chunk_size", 64), cu_seqlens=x.get("cu_seqlens"),
                        initial_state=x.get("initial_state"), dfinal_state=dfinal, segments=segments)
