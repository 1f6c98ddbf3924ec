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

from . import backward, forward, saved_size
from .inputs import WORKLOADS, make_inputs


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="fwdbwd_bf16_B4_T4096_H32_D128", choices=sorted(WORKLOADS))
    ap.add_argument("--B", type=int)
    ap.add_argument("--T", type=int)
    ap.add_argument("--H", type=int)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--fwd-only", action="store_true", help="skip the backward of a fwd+bwd workload")
    ap.add_argument("--saved", action="store_true", help="forward keeps the per-chunk record for the backward")
    a = ap.parse_args(argv)
    w = WORKLOADS[a.workload]
    over = {k: v for k, v in (("B", a.B), ("T", a.T), ("H", a.H)) if v is not None}
    if over:
        if w.varlen and ("B" in over or "T" in over):
            raise SystemExit("varlen workloads keep their packed length")
        w = dataclasses.replace(w, **over)
    dev = torch.device("cuda:0")
    x = make_inputs(w, device=dev)
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=x["chunk_size"],
              cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    run_bwd = w.backward and not a.fwd_only
    saved = None
    if run_bwd and a.saved:
        nb = saved_size(x["q"], x["v"], x["cu_seqlens"], x["chunk_size"])
        if nb == 0:
            raise SystemExit("this workload has no saved-record path")
        saved = torch.empty(nb, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(a.iters):
        forward(*[x[n] for n in names], output_final_state=w.final_state, saved=saved, **kw)
        if run_bwd:
            backward(*[x[n] for n in names], x["dout"], saved=saved, **kw)
    ev[1].record()
    torch.cuda.synchronize()
    print(f"workload={w.name} B={w.B} T={w.T} H={w.H} bwd={run_bwd} saved={saved is not None} iters={a.iters} "
          f"ms_per_iter={ev[0].elapsed_time(ev[1]) / max(1, a.iters):.3f}")


if __name__ == "__main__":
    main()
