"""Seeded synthetic inputs for the KDA workloads.

This module only draws random numbers: it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can take their inputs
from it.  Draws happen on the CPU with numpy's PCG64 in a fixed order
(lengths -> q -> k -> v -> g_raw -> beta_raw -> a_log -> dt_bias ->
initial_state -> dout), in float32, then the activations are cast to the
workload's dtype with torch (round to nearest even for bf16).

Distributions (the workloads quoted for this kernel):
  q, k, v, g_raw, beta_raw ~ N(0, 1); a_log ~ U(0, ln 16);
  dt_bias ~ N(0, 0.1^2); initial_state ~ N(0, 0.02^2); dout ~ N(0, 1);
  lower_bound = -5; scale = 1/sqrt(K).
The second argument of N(mean, x) is read as a standard deviation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str = "bf16"            # "bf16" or "fp32": dtype of q, k, v, g_raw, beta_raw, out, dout
    chunk_size: int = 64
    varlen: bool = False           # pack documents of random length into B=1, T tokens
    len_lo: int = 64
    len_hi: int = 4096
    initial_state: bool = False
    final_state: bool = False
    backward: bool = False
    lower_bound: float = -5.0
    g_mean: float = 0.0            # mean of g_raw (a "mild gate" variant shifts it negative)
    seed: int = 0
    Hk: int = 0                    # key heads of q, k (0: Hk = H); H value heads, H a multiple of Hk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.K)

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The five quoted workloads.
WORKLOADS = {
    "fwd_fp32_T256_H2_D64": Workload("fwd_fp32_T256_H2_D64", B=1, T=256, H=2, K=64, V=64, dtype="fp32"),
    "fwd_bf16_B2_T2048_H16_D128": Workload("fwd_bf16_B2_T2048_H16_D128", B=2, T=2048, H=16, K=128, V=128),
    "varlen_fwd_bf16_T16384_H32_D128": Workload("varlen_fwd_bf16_T16384_H32_D128", B=1, T=16384, H=32,
                                                K=128, V=128, varlen=True),
    "long_fwd_bf16_T65536_H32_D128": Workload("long_fwd_bf16_T65536_H32_D128", B=1, T=65536, H=32, K=128,
                                              V=128, initial_state=True, final_state=True),
    "fwdbwd_bf16_B4_T4096_H32_D128": Workload("fwdbwd_bf16_B4_T4096_H32_D128", B=4, T=4096, H=32, K=128,
                                              V=128, backward=True),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def draw_lengths(rng: np.random.Generator, total: int, lo: int, hi: int) -> list[int]:
    """Document lengths ~ U{lo..hi} drawn until they cover ``total``; the last is truncated."""
    lens: list[int] = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return lens


def make_inputs(w: Workload, device: str | torch.device = "cpu",
                lengths: Optional[list[int]] = None) -> dict:
    """Draw one batch for workload ``w``.

    Returns a dict of torch tensors on ``device``: q, k [B, T, Hk, K]; g_raw [B, T, H, K];
    v [B, T, H, V]; beta_raw [B, T, H]; a_log [H] fp32; dt_bias [H*K] fp32;
    cu_seqlens int32 [N+1] or None; initial_state fp32 [N, H, K, V] or None;
    dout [B, T, H, V] or None; plus the scalars scale, lower_bound, chunk_size.
    ``lengths`` overrides the random document lengths of a varlen workload.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    Hk = w.Hk or H
    cu = None
    if w.varlen:
        if lengths is None:
            lengths = draw_lengths(rng, B * T, w.len_lo, w.len_hi)
        assert B == 1 and sum(lengths) == T, "varlen workloads pack B=1 rows of T tokens"
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    n_seq = (len(cu) - 1) if cu is not None else B
    dt = _torch_dtype(w.dtype)

    def normal(shape, std=1.0, mean=0.0):
        x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(shape)
        if std != 1.0:
            x *= np.float32(std)
        if mean != 0.0:
            x += np.float32(mean)
        return x

    def act(x):
        return torch.from_numpy(x).to(dt).to(device)

    out = {}
    out["q"] = act(normal((B, T, Hk, K)))
    out["k"] = act(normal((B, T, Hk, K)))
    out["v"] = act(normal((B, T, H, V)))
    out["g_raw"] = act(normal((B, T, H, K), mean=w.g_mean))
    out["beta_raw"] = act(normal((B, T, H)))
    out["a_log"] = torch.from_numpy(rng.uniform(0.0, math.log(16.0), H).astype(np.float32)).to(device)
    out["dt_bias"] = torch.from_numpy(normal((H * K,), std=0.1)).to(device)
    out["initial_state"] = (torch.from_numpy(normal((n_seq, H, K, V), std=0.02)).to(device)
                            if w.initial_state else None)
    out["dout"] = act(normal((B, T, H, V))) if w.backward else None
    out["cu_seqlens"] = torch.from_numpy(cu).to(device) if cu is not None else None
    out["scale"] = w.scale
    out["lower_bound"] = w.lower_bound
    out["chunk_size"] = w.chunk_size
    return out
