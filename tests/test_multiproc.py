"""Multi-process host logic of the replica path (bench.py), world size 2 over gloo on the CPU.

The kernel path shards over (segment, head) units with no exchange, so N GPUs run independent
replicas: each rank draws its own inputs (seed + rank), the only collectives are the barrier
around the timed region and the max-over-ranks of the timings.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    from gated_delta_rule_sm_gb300.inputs import WORKLOADS, make_inputs
    import dataclasses

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        assert (r, wsz, local) == (rank, world, rank)
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 + rank, world)
        w = dataclasses.replace(WORKLOADS["fwd_fp32_T256_H2_D64"], seed=WORKLOADS["fwd_fp32_T256_H2_D64"].seed + rank)
        x = make_inputs(w)
        out.put((rank, slowest, float(x["q"].double().sum())))
    finally:
        dist.destroy_process_group()


def test_replicas_world2_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    # max over ranks is the slowest rank's time on every rank
    assert [r[1] for r in res] == [11.0, 11.0]
    # each replica draws its own shard of inputs
    assert res[0][2] != res[1][2]


def test_single_rank_helpers_are_identities():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)   # no process group needed


def test_reference_arm_runs_on_rank0_only():
    """Under torchrun only rank 0 times the oracle; the other ranks exit 0 without output."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
