"""The benchmark's multi-rank host logic on CPU with the gloo backend and two
ranks: each rank gets its own units (weak scaling, no collective on the
path), the timings are reduced with a maximum over ranks, and the job value
counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from recallable_kv_cache_gb300 import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        base = synth.scaled(synth.WORKLOADS["layer_32k"], units=2, L=16 + 64, decode_steps=4)
        w = bench.rank_workload(base, rank, world)
        keys = synth.unit_keys(w, 0)
        # the slowest rank decides: rank r reports times (r + 1, 10 - r, 3)
        step, prefill, decode = bench.max_over_ranks([rank + 1.0, 10.0 - rank, 3.0], world, device="cpu")
        gathered = [None] * world
        dist.all_gather_object(gathered, (w.seed, float(keys.float().sum())))
        dist.barrier()
        if rank == 0:
            out.put(dict(maxes=(step, prefill, decode), seeds=[g[0] for g in gathered],
                         sums=[g[1] for g in gathered],
                         value=bench.job_value(world, w.decode_steps, step)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling_and_max_timing():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = out.get()
    assert list(res["maxes"]) == [2.0, 10.0, 3.0]
    seeds, sums = res["seeds"], res["sums"]
    assert seeds[0] != seeds[1] and sums[0] != sums[1]  # own units, own data
    assert res["value"] == pytest.approx(2 * 4 / (2.0 / 1000.0))


def test_single_rank_needs_no_process_group():
    base = synth.WORKLOADS["layer_32k"]
    assert bench.rank_workload(base, 0, 1) is base
    assert bench.max_over_ranks([1.0, 2.0], 1) == [1.0, 2.0]
    assert bench.job_value(1, 1024, 50.0) == pytest.approx(1024 / 0.05)
