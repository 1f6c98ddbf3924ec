"""GPU parity of the gated output norm (``kda_gated_norm_fwd`` / ``_bwd``) against the fp64 oracle.

This file is collected after the recurrence's parity tests, so that a failure here leaves them run.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import gated_delta_rule_sm_gb300 as kda  # noqa: E402
from kda_cases import f64, rel_err, tol  # noqa: E402

DEV = "cuda:0"


def _case(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o = torch.randn(shape, generator=g).to(dt)
    gate = torch.randn(shape, generator=g).to(dt)
    w = torch.rand((shape[-1],), generator=g) + 0.5
    dy = torch.randn(shape, generator=g).to(dt)
    return o, gate, w, dy


@pytest.mark.parametrize("shape,dtype", [((2, 150, 3, 128), "bf16"), ((1, 77, 2, 64), "fp32"),
                                         ((1, 33, 5, 48), "fp32"), ((3, 10, 1, 256), "bf16"), ((1, 1, 1, 16), "fp32")])
def test_gated_norm_fwd_bwd(shape, dtype):
    o, gate, w, dy = _case(shape, dtype, seed=sum(shape))
    y = kda.gated_norm(o.to(DEV), gate.to(DEV), w.to(DEV), eps=1e-6)
    g = kda.gated_norm_backward(o.to(DEV), gate.to(DEV), w.to(DEV), dy.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ry = oracle.gated_norm_fwd(f64(o), f64(gate), f64(w), 1e-6)
    rg = oracle.gated_norm_bwd(f64(o), f64(gate), f64(w), 1e-6, f64(dy))
    assert y.dtype == o.dtype and y.shape == o.shape
    assert rel_err(y, ry, dtype) <= tol(dtype)
    # the gradients are fp32 results computed from the exact (bf16 or fp32) inputs: fp32 bound whatever
    # the activation dtype
    for n in ("do", "dgate", "dweight"):
        e = rel_err(g[n], rg[n], "fp32")
        assert e <= tol("fp32"), (n, e)


def test_gated_norm_at_the_training_shape():
    """B4 T4096 H32 V128 bf16, the fwd+bwd workload's output: every row against the oracle; the backward
    twice, bit-identical (dweight sums in a fixed order)."""
    o, gate, w, dy = _case((4, 4096, 32, 128), "bf16", seed=90)
    od, gd, wd, dyd = (t.to(DEV) for t in (o, gate, w, dy))
    y = kda.gated_norm(od, gd, wd)
    g1 = kda.gated_norm_backward(od, gd, wd, dyd)
    g2 = kda.gated_norm_backward(od, gd, wd, dyd)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    for n in ("do", "dgate", "dweight"):
        assert torch.equal(g1[n], g2[n]), n
    ry = oracle.gated_norm_fwd(f64(o), f64(gate), f64(w), 1e-6)
    rg = oracle.gated_norm_bwd(f64(o), f64(gate), f64(w), 1e-6, f64(dy))
    assert rel_err(y, ry, "bf16") <= tol("bf16")
    for n in ("do", "dgate", "dweight"):
        e = rel_err(g1[n], rg[n], "fp32")
        assert e <= tol("fp32"), (n, e)
