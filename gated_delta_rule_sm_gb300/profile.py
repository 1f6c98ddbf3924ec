"""Run the KDA library a fixed number of times on one workload, for ncu captures.

    python -m gated_delta_rule_sm_gb300.profile --workload fwdbwd_bf16_B4_T4096_H32_D128 --iters 3
    python -m gated_delta_rule_sm_gb300.profile --workload fwdbwd_bf16_B4_T4096_H32_D128 --B 1 --iters 2 --saved

``--B/--T/--H`` shrink a named workload (same distributions, same seed) so a
capture with many metric passes stays small.  Inputs are drawn once and kept
on the device; each iteration runs the forward, and the backward when the
workload has one.  ``--saved`` runs the training pair the benchmark times (a forward that keeps the
per-chunk record, then the backward that reads it) instead of two independent calls.  Prints one line with the mean CUDA-event time per
iteration (a number taken under a profiler is not a benchmark value).
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import _lib, backward, forward, saved_size
from .inputs import WORKLOADS, make_inputs


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="fwdbwd_bf16_B4_T4096_H32_D128", choices=sorted(WORKLOADS))
    ap.add_argument("--B", type=int)
    ap.add_argument("--T", type=int)
    ap.add_argument("--H", type=int)
    ap.add_argument("--D", type=int, help="head size K = V (64 or 128)")
    ap.add_argument("--dtype", choices=("bf16", "fp32"), help="activation dtype (fp32 runs the SIMT path)")
    ap.add_argument("--Hk", type=int, help="key heads (H a multiple of it; grouped heads)")
    ap.add_argument("--final-state", action="store_true", help="also write the final state")
    ap.add_argument("--initial-state", action="store_true", help="also read an initial state")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=0, help="untimed iterations before the timed ones")
    ap.add_argument("--kernels", action="store_true", help="also print each kernel's mean time (library events)")
    ap.add_argument("--fwd-only", action="store_true", help="skip the backward of a fwd+bwd workload")
    ap.add_argument("--saved", action="store_true", help="forward keeps the per-chunk record for the backward")
    ap.add_argument("--segments", type=int, default=0,
                    help="forward and backward through kda_fwd_segmented / kda_bwd_segmented, rows cut into "
                         "pieces of 1 / segments of a row")
    ap.add_argument("--gate", default="lower_bounded", choices=("lower_bounded", "softplus"),
                    help="gate activation (softplus: the unbounded gate)")
    ap.add_argument("--gated-norm", action="store_true",
                    help="instead time the gated output norm (forward and backward) on the workload's [B, T, H, V] output")
    ap.add_argument("--short-conv", type=int, default=0, metavar="W",
                    help="instead time the W-tap short convolution + SiLU prologue on a q-shaped [B, T, H*K] tensor")
    a = ap.parse_args(argv)
    w = WORKLOADS[a.workload]
    over = {k: v for k, v in (("B", a.B), ("T", a.T), ("H", a.H), ("dtype", a.dtype), ("Hk", a.Hk), ("K", a.D),
                              ("V", a.D)) if v is not None}
    if a.final_state:
        over["final_state"] = True
    if a.initial_state:
        over["initial_state"] = True
    if over:
        if w.varlen and ("B" in over or "T" in over):
            raise SystemExit("varlen workloads keep their packed length")
        w = dataclasses.replace(w, **over)
    dev = torch.device("cuda:0")
    if a.short_conv:
        _time_short_conv(w, a.short_conv, a.iters, dev)
        return
    if a.gated_norm:
        _time_gated_norm(w, a.iters, dev)
        return
    x = make_inputs(w, device=dev)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], gate=a.gate, chunk_size=x["chunk_size"],
              cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    run_bwd = w.backward and not a.fwd_only
    saved = None
    if run_bwd and a.saved:
        nb = saved_size(x["q"], x["v"], x["cu_seqlens"], x["chunk_size"], a.gate)
        if nb == 0:
            raise SystemExit("this workload has no saved-record path")
        saved = torch.empty(nb, dtype=torch.uint8, device=dev)
    if a.segments:
        kw["segments"] = a.segments
        if saved is not None:
            raise SystemExit("--segments runs without --saved")

    def step():
        forward(*[x[n] for n in names], output_final_state=w.final_state, saved=saved, **kw)
        if run_bwd:
            backward(*[x[n] for n in names], x["dout"], saved=saved, **kw)

    for _ in range(a.warmup):
        step()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    if a.kernels:
        _lib.timing_begin(64 * a.iters)
    ev[0].record()
    for _ in range(a.iters):
        step()
    ev[1].record()
    torch.cuda.synchronize()
    if a.kernels:
        per: dict = {}
        for name, ms in _lib.timing_end(64 * a.iters):
            per[name] = per.get(name, 0.0) + ms
        print("  ".join(f"{k}={v / max(1, a.iters):.3f}ms" for k, v in per.items()))
    print(f"workload={w.name} B={w.B} T={w.T} H={w.H} gate={a.gate} segments={a.segments} bwd={run_bwd} "
          f"saved={saved is not None} "
          f"iters={a.iters} "
          f"ms_per_iter={ev[0].elapsed_time(ev[1]) / max(1, a.iters):.3f}")


def _time_gated_norm(w, iters: int, dev) -> None:
    """Forward and backward of the output epilogue on a [B, T, H, V] tensor of the workload's dtype."""
    from . import gated_norm, gated_norm_backward
    g = torch.Generator().manual_seed(w.seed)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    shape = (w.B, w.T, w.H, w.V)
    o, gate, dy = (torch.randn(shape, generator=g).to(dt).to(dev) for _ in range(3))
    wt = (torch.rand((w.V,), generator=g) + 0.5).to(dev)
    y = torch.empty_like(o)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(3):
        gated_norm(o, gate, wt, out=y)
        gated_norm_backward(o, gate, wt, dy)
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(iters):
        gated_norm(o, gate, wt, out=y)
    ev[1].record()
    for _ in range(iters):
        gated_norm_backward(o, gate, wt, dy)
    ev[2].record()
    torch.cuda.synchronize()
    e, n = o.element_size(), o.numel()
    f_ms = ev[0].elapsed_time(ev[1]) / iters
    b_ms = ev[1].elapsed_time(ev[2]) / iters
    # algorithmic bytes: forward reads o, gate and writes y; backward reads o, gate, dy and writes fp32 do, dgate
    fb, bb = n * 3 * e, n * (3 * e + 8)
    print(f"gated_norm B={w.B} T={w.T} H={w.H} V={w.V} dtype={w.dtype} fwd_ms={f_ms:.4f} fwd_GBs={fb / f_ms / 1e6:.0f} "
          f"bwd_ms={b_ms:.4f} bwd_GBs={bb / b_ms / 1e6:.0f}")


def _time_short_conv(w, W: int, iters: int, dev) -> None:
    """Forward and backward of the prologue convolution on a [B, T, H*K] activation of the workload."""
    from . import short_conv, short_conv_backward
    g = torch.Generator().manual_seed(w.seed)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    C = w.H * w.K
    x = torch.randn((w.B, w.T, C), generator=g).to(dt).to(dev)
    dy = torch.randn((w.B, w.T, C), generator=g).to(dt).to(dev)
    wt = (0.5 * torch.randn((C, W), generator=g)).to(dev)
    b = (0.1 * torch.randn((C,), generator=g)).to(dev)
    y = torch.empty_like(x)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(3):
        short_conv(x, wt, b, out=y)
        short_conv_backward(x, wt, b, dy)
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(iters):
        short_conv(x, wt, b, out=y)
    ev[1].record()
    for _ in range(iters):
        short_conv_backward(x, wt, b, dy)
    ev[2].record()
    torch.cuda.synchronize()
    e = x.element_size()
    n = x.numel()
    f_ms = ev[0].elapsed_time(ev[1]) / iters
    b_ms = ev[1].elapsed_time(ev[2]) / iters
    # algorithmic bytes: forward reads x, writes y; backward reads x, dy, writes fp32 dx
    fb, bb = n * 2 * e, n * (2 * e + 4)
    print(f"short_conv W={W} B={w.B} T={w.T} C={C} dtype={w.dtype} fwd_ms={f_ms:.4f} fwd_GBs={fb / f_ms / 1e6:.0f} "
          f"bwd_ms={b_ms:.4f} bwd_GBs={bb / b_ms / 1e6:.0f}")


if __name__ == "__main__":
    main()
