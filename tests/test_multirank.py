"""The multi-process host logic of bench.py, on CPU with two gloo ranks.

The attention path shards over (batch, head) with no exchange step, so a
run on N GPUs is N independent replicas: each rank owns its own copy of the
workload, the only collective is the max-over-ranks of the step time, and
whole-job throughput is the sum of the ranks' work over that time.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    wl = bench.rank_workload(bench.WORKLOAD, r)
    ms = bench.max_over_ranks(1.5 + 2.0 * rank, dist, "cpu")
    out.put((r, w, local, wl.seed, wl.B, wl.H, wl.N_q, ms))
    dist.destroy_process_group()


def test_two_ranks_independent_replicas_and_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, s0, *shape0, ms0), (r1, w1, l1, s1, *shape1, ms1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert shape0 == shape1                  # the same per-rank workload (weak scaling) ...
    assert s0 != s1                          # ... on independent inputs
    assert ms0 == ms1 == 3.5                 # every rank reports the slowest rank's time


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        warmup, steps, ref_budget = 3, 1, 60.0
    assert bench.run_reference(Args()) == 0   # returns at once: no oracle work on rank 1
