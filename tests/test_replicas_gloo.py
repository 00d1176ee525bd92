"""Multi-process logic of the benchmark on CPU (gloo, world size 2).

The decode path shards as independent replicas: each rank serves its own
batch of sequences and nothing crosses ranks on the data path.  What crosses
ranks is measurement only -- the barrier around the timed region and the
maximum of the ranks' times -- and that is what these tests run, as two gloo
processes on 127.0.0.1.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from learned_kv_cache_eviction_b300 import workload as W


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        dist.barrier()
        ms = bench.max_over_ranks(dist, local_ms, "cpu")
        wl = bench.replica_workload(W.WORKLOADS["tiny"], rank)
        k, _, lg = W.kv_range(wl, 0, 0, 8)
        q.put((rank, ms, wl.seed, float(k.float().sum()), float(lg.sum()),
               bench.job_tokens_per_s(wl.B, 10, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_draw_their_own_inputs():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    (r0, ms0, seed0, ksum0, lsum0, v0), (r1, ms1, seed1, ksum1, lsum1, v1) = res
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 5.0                          # the slowest rank's time on every rank
    assert seed0 != seed1 and ksum0 != ksum1 and lsum0 != lsum1  # independent sequences per rank
    assert v0 == v1 == pytest.approx(1 * 10 * 2 / 5e-3)         # tokens of both ranks / slowest time


def test_single_process_helpers():
    assert bench.max_over_ranks(None, 2.5, "cpu") == 2.5
    wl = W.WORKLOADS["qwen3-8b"]
    assert bench.replica_workload(wl, 0) is wl
    assert bench.replica_workload(wl, 3).seed == wl.seed + 3000
    assert bench.job_tokens_per_s(32, 100, 1, 10.0) == pytest.approx(3.2e5)
