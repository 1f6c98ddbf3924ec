#!/usr/bin/env python
"""KDA benchmark on GB300: tokens/s of one step of the hot path, with its roofline.

A step is one pass of the whole path over one batch of synthetic input: the
forward (gate / beta / L2-norm prologue, intra-chunk WY transform,
inter-chunk state chain, output) followed by the backward (reverse state
chain, per-chunk gradients, prologue backward and parameter reductions), on
the fwd+bwd workload B=4, T=4096, H=32, K=V=128, bf16 inputs, fp32 state and
gradients.  ``--workload`` selects another workload (forward-only ones time
the forward alone).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "fwdbwd_bf16_B4_T4096_H32_D128"
# the five quoted workloads, in order; the default one is the headline, the others go in per_config
WORKLOAD_NAMES = ("fwd_fp32_T256_H2_D64", "fwd_bf16_B2_T2048_H16_D128", "varlen_fwd_bf16_T16384_H32_D128",
                  "long_fwd_bf16_T65536_H32_D128", "fwdbwd_bf16_B4_T4096_H32_D128")
METRIC = "KDA fwd(+bwd) tokens/sec on 1 GB300"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ algorithmic work per token-head

def algorithmic(K: int, V: int, C: int = 64, act_bytes: int = 2) -> dict:
    """Bytes and FLOPs the method must move / compute per token-head (triangles counted once).

    forward FLOPs  = 3CK + 2CV + 6KV + C^2/3   (intra: 3CK + CV + C^2/3, chain: 6KV + CV)
    forward bytes  = act_bytes * (3K + K... ) : reads q, k, g_raw (K each), v (V), beta (1), writes o (V)
    backward bytes = re-read q, k, v, g, beta + read dout + write fp32 dq, dk, dg, dv, dbeta
    backward FLOPs ~ 2 x forward.
    """
    fwd_read = act_bytes * (3 * K + V + 1)
    fwd_write = act_bytes * V
    fwd_flops = 3 * C * K + 2 * C * V + 6 * K * V + C * C / 3
    bwd_bytes = fwd_read + act_bytes * V + 4 * (3 * K + V + 1)
    return dict(fwd_bytes=fwd_read + fwd_write, fwd_read=fwd_read, fwd_write=fwd_write, fwd_flops=fwd_flops,
                intra_flops=3 * C * K + C * V + C * C / 3, chain_flops=6 * K * V + C * V,
                bwd_bytes=bwd_bytes, bwd_flops=2 * fwd_flops)


def kernel_work(name: str, w, units: float) -> tuple[float, float]:
    """(algorithmic bytes, FLOPs) one launch of kernel ``name`` is responsible for, ``units`` = token-heads."""
    a = algorithmic(w.K, w.V, act_bytes=2 if w.dtype == "bf16" else 4)
    table = {
        "kda_intra_simt": (a["fwd_read"], a["intra_flops"]),
        "kda_chain_fwd_simt": (a["fwd_write"], a["chain_flops"]),
        "kda_intra_tc": (a["fwd_read"], a["intra_flops"]),
        "kda_chain_fwd_tc": (a["fwd_write"], a["chain_flops"]),
        "kda_chain_bwd_simt": (0.0, a["chain_flops"]),
        "kda_chain_bwd_tc": (0.0, a["chain_flops"]),
        "kda_bwd_pre": (0.0, 0.0),
        # the per-chunk gradient kernels read dout and write every fp32 gradient
        "kda_grad_simt": (a["bwd_bytes"] - a["fwd_read"], a["bwd_flops"] - a["chain_flops"] - a["intra_flops"]),
        "kda_grad_tc": (a["bwd_bytes"] - a["fwd_read"], a["bwd_flops"] - a["chain_flops"] - a["intra_flops"]),
    }
    b, f = table.get(name, (0.0, 0.0))
    return b * units, f * units


# DRAM bytes (read + write) per token-head per launch, from one-kernel ncu captures of the current
# kernels on shortened shapes of the same workloads (B=1 T=4096 H=32 for the training step, T=8192
# H=32 for the long forward).  Per-chunk kernels move the same bytes per chunk-head at any size, so
# the figure scales with the token-heads of a launch.  An entry is removed when its kernel changes and
# has not been captured again.
PROFILED_TRAFFIC = {
    ("kda_grad_tc", True): 8353.0,
    ("kda_intra_tc", False): 2222.0,   # forward record only (forward-only workloads; intra2_kernel)
    ("kda_intra_tc", True): 6859.0,    # forward that keeps the backward record, once per training step
}


def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            out = {"source": "measured"}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                out[k] = float(v) if v is not None else FALLBACK_PEAKS[k]
            return out
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (identity when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ CPU baseline (oracle)

def cpu_baseline(w, x_cpu: dict, budget_s: float = 15.0) -> dict:
    """The fp64 oracle, as it stands, on a bounded sample of (segment, head) pairs of the workload."""
    import numpy as np

    import oracle
    cores = os.cpu_count() or 1
    K = w.K
    heads_total = w.H
    rows = 1
    f64 = lambda t: t.detach().to(dtype=__import__("torch").float64).cpu().numpy()
    # pairs: the first `rows` batch rows, first `nh` heads; grow heads, then rows, until the budget is met
    T = w.T
    nh = 1
    sample_desc = ""
    elapsed = 0.0
    while True:
        heads = list(range(min(nh, heads_total)))
        sl = lambda t, last=None: t[:rows][:, :, heads] if t is not None else None
        args = [f64(sl(x_cpu["q"])), f64(sl(x_cpu["k"])), f64(sl(x_cpu["v"])), f64(sl(x_cpu["g_raw"])),
                f64(x_cpu["beta_raw"][:rows][:, :, heads]), f64(x_cpu["a_log"][heads]),
                f64(x_cpu["dt_bias"].view(-1, K)[heads].reshape(-1))]
        S0 = f64(x_cpu["initial_state"][:rows][:, heads]) if x_cpu.get("initial_state") is not None else None
        cu = None
        if x_cpu.get("cu_seqlens") is not None:
            cu = x_cpu["cu_seqlens"].numpy().astype(np.int64)
        t0 = time.perf_counter()
        oracle.kda_fwd(*args, scale=w.scale, lower_bound=w.lower_bound, cu_seqlens=cu, initial_state=S0,
                       nthreads=cores)
        if w.backward:
            oracle.kda_bwd(*args, f64(x_cpu["dout"][:rows][:, :, heads]), scale=w.scale,
                           lower_bound=w.lower_bound, cu_seqlens=cu, initial_state=S0, nthreads=cores)
        elapsed = time.perf_counter() - t0
        sample_desc = (f"{'fwd+bwd' if w.backward else 'fwd'} of batch rows 0..{rows - 1} ({rows} of {w.B}), "
                       f"heads 0..{len(heads) - 1} ({len(heads)} of {heads_total}), all {T} tokens per row")
        if elapsed * 2 > budget_s:
            break
        if len(heads) < heads_total:
            nh = min(heads_total, max(nh * 2, int(nh * budget_s / max(elapsed, 1e-3) * 0.5)))
        elif rows < w.B and cu is None:
            rows = min(w.B, max(rows + 1, int(rows * budget_s / max(elapsed, 1e-3) * 0.5)))
        else:
            break
    tok_heads = rows * T * len(heads)
    value = tok_heads / heads_total / elapsed          # tokens/s, a token carrying all H heads
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample_desc,
            "seconds": elapsed}


# ------------------------------------------------------------------ the other workloads, same process

def step_roofline_of(w, ms_step: float, peaks: dict) -> dict:
    a = algorithmic(w.K, w.V, act_bytes=2 if w.dtype == "bf16" else 4)
    step_bytes = w.tokens * w.H * (a["fwd_bytes"] + (a["bwd_bytes"] if w.backward else 0))
    state_bytes = 4 * w.H * w.K * w.V * (w.B if not w.varlen else 0) * (int(w.initial_state) + int(w.final_state))
    step_bytes += state_bytes
    step_flops = w.tokens * w.H * (a["fwd_flops"] + (a["bwd_flops"] if w.backward else 0))
    roof_s = max(step_bytes / (peaks["hbm_gbs"] * 1e9), step_flops / (peaks["bf16_tflops"] * 1e12))
    return {"roofline_ms": roof_s * 1e3, "frac": roof_s / (ms_step / 1e3), "bytes": step_bytes,
            "flops": step_flops, "peak_source": peaks["source"]}


def time_workload(name: str, dev, steps: int, warmup: int, peaks: dict) -> dict:
    """Device time of one workload's step (forward, or forward + backward), timed step by step with CUDA
    events on the launching stream and L2 flushed (a 256 MiB write) before every step, since the smaller
    workloads' inputs fit in L2.  Returns ms per step, tokens/s, the step roofline fraction, the
    dominant kernel and the clocks seen while timing."""
    import torch

    import gated_delta_rule_sm_gb300 as kda
    from gated_delta_rule_sm_gb300 import _lib
    from gated_delta_rule_sm_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    x = {k: (v.to(dev) if hasattr(v, "to") else v) for k, v in make_inputs(w, device="cpu").items()}
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=x["chunk_size"],
              cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])
    outs = {}
    nsaved = kda.saved_size(x["q"], x["v"], x["cu_seqlens"]) if w.backward else 0
    saved = torch.empty(nsaved, dtype=torch.uint8, device=dev) if nsaved > 0 else None

    def step():
        o, fs = kda.forward(*[x[n] for n in names], output_final_state=w.final_state, out=outs.get("out"),
                            final_state=outs.get("fs"), saved=saved, **kw)
        outs["out"], outs["fs"] = o, fs
        if w.backward:
            outs["grads"] = kda.backward(*[x[n] for n in names], x["dout"], grads=outs.get("grads"), saved=saved,
                                         **kw)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert kda.device_status() == 0, f"device status word set during warm-up of {name}"
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    _lib.timing_begin(64 * steps)
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    launches = _lib.timing_end(64 * steps)
    clk = clocks.stop()
    assert kda.device_status() == 0
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    per = {}
    for kname, kms in launches:
        per[kname] = per.get(kname, 0.0) + kms
    tot = sum(per.values())
    dom = max(per.items(), key=lambda kv: kv[1])[0] if per else None
    del x, outs, saved, flush
    torch.cuda.empty_cache()
    return {"workload": name, "ms": ms, "tokens_per_s": w.tokens / (ms / 1e3),
            "step_roofline": step_roofline_of(w, ms, peaks), "backward": w.backward,
            "dominant_kernel": dom, "dominant_share": (per[dom] / tot) if dom else None,
            "kernels_ms_per_step": {k: v / steps for k, v in sorted(per.items(), key=lambda kv: -kv[1])},
            "l2": "flushed before every step", "clocks": clk}


# ------------------------------------------------------------------ our implementation

def run_ours(args, w):
    import torch

    import gated_delta_rule_sm_gb300 as kda
    from gated_delta_rule_sm_gb300 import _lib
    from gated_delta_rule_sm_gb300.inputs import make_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.load()
    import dataclasses
    wr = dataclasses.replace(w, seed=w.seed + rank)
    x_cpu = make_inputs(wr, device="cpu")
    x = {k: (v.to(dev) if hasattr(v, "to") else v) for k, v in x_cpu.items()}
    names = ("q", "k", "v", "g_raw", "beta_raw", "a_log", "dt_bias")
    kw = dict(scale=x["scale"], lower_bound=x["lower_bound"], chunk_size=x["chunk_size"],
              cu_seqlens=x["cu_seqlens"], initial_state=x["initial_state"])

    outs = {}
    # a training step: the forward keeps the per-chunk quantities the backward would rebuild
    nsaved = kda.saved_size(x["q"], x["v"], x["cu_seqlens"]) if w.backward else 0
    saved = torch.empty(nsaved, dtype=torch.uint8, device=dev) if nsaved > 0 else None

    def step(inp):
        o, fs = kda.forward(*[inp[n] for n in names], output_final_state=w.final_state,
                            out=outs.get("out"), final_state=outs.get("fs"), saved=saved, **kw)
        outs["out"], outs["fs"] = o, fs
        if w.backward:
            outs["grads"] = kda.backward(*[inp[n] for n in names], inp["dout"], grads=outs.get("grads"),
                                         saved=saved, **kw)

    for _ in range(args.warmup):
        step(x)
    torch.cuda.synchronize()
    assert kda.device_status() == 0, "device status word set during warm-up"

    # ---- device-resident timed region.  Inputs larger than L2 need no flush between steps; a workload
    # that fits in L2 is timed step by step with a 256 MiB write (L2 flush) before every step.
    peaks = read_peaks()
    fits_l2 = step_roofline_of(w, 1.0, peaks)["bytes"] < 2 * 129e6
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if fits_l2 else None
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world, dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _lib.timing_begin(64 * args.steps)
    if fits_l2:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            step(x)
            e1.record(stream)
    else:
        ev0.record(stream)
        for _ in range(args.steps):
            step(x)
        ev1.record(stream)
    torch.cuda.synchronize()
    launches = _lib.timing_end(64 * args.steps)
    barrier(world, dev)
    clk = clocks.stop()
    ms_total = sum(e0.elapsed_time(e1) for e0, e1 in evs) if fits_l2 else ev0.elapsed_time(ev1)
    ms_step = max_over_ranks(ms_total / args.steps, world, dev)
    del flush
    assert kda.device_status() == 0

    # ---- end to end: pinned host inputs -> device, the C-ABI calls, results -> pinned host.
    # Every step copies its inputs in and its results out.  As a training loop would, the copies run
    # on their own streams, double-buffered, so step i+1's inputs arrive and step i-1's results
    # leave while step i computes; the timed region spans all of it.
    in_names = list(names) + (["dout"] if w.backward else [])
    if x_cpu.get("initial_state") is not None:
        in_names.append("initial_state")
    if x_cpu.get("cu_seqlens") is not None:
        in_names.append("cu_seqlens")
    host_in = {n: x_cpu[n].pin_memory() for n in in_names}
    dev_in = [{n: torch.empty_like(x[n]) for n in in_names} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())

    def result_tensors(o):
        res = [o["out"]]
        if o.get("fs") is not None:
            res.append(o["fs"])
        if w.backward:
            res += [t for t in o["grads"].values() if t is not None]
        return res

    outs_b = [outs, {"out": torch.empty_like(outs["out"]),
                     "fs": torch.empty_like(outs["fs"]) if outs.get("fs") is not None else None,
                     "grads": ({k: (torch.empty_like(t) if t is not None else None)
                                for k, t in outs["grads"].items()} if w.backward else None)}]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in result_tensors(outs)]
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b landed
    ev_used = [torch.cuda.Event() for _ in range(2)]   # compute on buffer b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # results of buffer b copied out
    for e in ev_used + ev_out:
        e.record(stream)

    def e2e_step(i):
        b = i & 1
        ob = outs_b[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[b])                 # step i-2 is done reading this input buffer
            for n in in_names:
                dev_in[b][n].copy_(host_in[n], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])                    # step i-2's results in this buffer have left
        inp = dict(x, **dev_in[b])
        kda.forward(*[inp[n] for n in names], output_final_state=w.final_state, out=ob["out"],
                    final_state=ob.get("fs"), scale=x["scale"], lower_bound=x["lower_bound"],
                    chunk_size=x["chunk_size"], cu_seqlens=inp.get("cu_seqlens"),
                    initial_state=inp.get("initial_state"), saved=saved)
        if w.backward:
            kda.backward(*[inp[n] for n in names], inp["dout"], grads=ob["grads"], scale=x["scale"],
                         lower_bound=x["lower_bound"], chunk_size=x["chunk_size"], cu_seqlens=inp.get("cu_seqlens"),
                         initial_state=inp.get("initial_state"), saved=saved)
        ev_used[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[b])
            for h, t in zip(host_out, result_tensors(ob)):
                h.copy_(t, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world, dev)
    ev0.record(stream)
    s_in.wait_event(ev0)
    s_out.wait_event(ev0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_event(ev_out[(args.steps - 1) & 1])    # the last step's results are on the host
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    for h, t in zip(host_out, result_tensors(outs_b[(args.steps - 1) & 1])):
        assert torch.equal(h, t.cpu()), "end-to-end results on the host differ from the device"

    tokens = w.tokens
    value = world * tokens / (ms_step / 1e3)

    # ---- dominant kernel roofline
    per = {}
    for name, ms in launches:
        d = per.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += ms
    dom = max(per.items(), key=lambda kv: kv[1][1])[0] if per else None
    roofline = None
    if dom is not None:
        n_launch, tot_ms = per[dom]
        avg_s = tot_ms / n_launch / 1e3
        units = w.tokens * w.H
        launches_per_step = n_launch / args.steps
        bytes_l, flops_l = kernel_work(dom, w, units / max(1.0, launches_per_step))
        hbm = peaks["hbm_gbs"]
        tfl = peaks["bf16_tflops"]
        t_bytes = bytes_l / (hbm * 1e9)
        t_flops = flops_l / (tfl * 1e12)
        if t_flops > t_bytes:
            roofline = {"bound": "tensor", "achieved": flops_l / avg_s / 1e12, "peak": tfl, "unit": "TFLOP/s"}
        else:
            roofline = {"bound": "hbm", "achieved": bytes_l / avg_s / 1e9, "peak": hbm, "unit": "GB/s"}
        roofline["frac"] = roofline["achieved"] / roofline["peak"]
        tpu = PROFILED_TRAFFIC.get((dom, bool(w.backward)))
        roofline["traffic"] = tpu * units / max(1.0, launches_per_step) if tpu is not None and w.K == 128 else None
        roofline["kernel"] = dom
        roofline["peak_source"] = peaks["source"]
        roofline["avg_launch_ms"] = tot_ms / n_launch
    step_roofline = step_roofline_of(w, ms_step, peaks)
    step_bytes = step_roofline["bytes"]
    kernels = {k: {"launches": v[0], "ms_total": v[1]} for k, v in sorted(per.items(), key=lambda kv: -kv[1][1])}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == "fp32" else "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                   "chunk_size": w.chunk_size, "backward": w.backward, "tokens_per_step": w.tokens,
                   "global_batch": w.B * world, "seq_len": w.T,
                   "parallelism": f"replicas x{world} (independent shards, no collective)",
                   "l2": "L2 flushed before every timed step" if fits_l2 else "inputs larger than L2 (no flush)"},
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": len(launches),
        "roofline": roofline,
        "step_roofline": step_roofline,
        "kernels": kernels,
        "clocks": clk,
    }
    if world == 1 and not args.no_per_config:
        # every other workload, timed in this process (forward-only workloads time the forward)
        del host_in, dev_in, outs_b, host_out, outs, saved, x
        torch.cuda.empty_cache()
        result["per_config"] = [time_workload(n, dev, args.config_steps, args.warmup, peaks)
                                for n in WORKLOAD_NAMES if n != w.name]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, x_cpu, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, w):
    """The fp64 CPU oracle, as it stands, on host cores: a bounded sample per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from gated_delta_rule_sm_gb300.inputs import make_inputs
    x_cpu = make_inputs(w, device="cpu")
    for _ in range(args.warmup):
        cpu_baseline(w, x_cpu, budget_s=0.5)
    vals = []
    base = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        base = cpu_baseline(w, x_cpu, budget_s=args.ref_budget)
        vals.append(base["value"])
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    ms_step = w.tokens / value * 1e3
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
                   "chunk_size": w.chunk_size, "backward": w.backward, "tokens_per_step": w.tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": base["cores"], "kind": "oracle",
                         "sample": base["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip timing the other workloads")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps per workload in per_config")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="seconds of oracle work per reference step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    from gated_delta_rule_sm_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
