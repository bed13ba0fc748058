"""The multi-GPU bench path on CPU: two gloo ranks.

Streams are independent, so N GPUs run N independent replicas of the
workload (weak scaling, no collective on the data path); the only exchange is
the max over ranks of the timed seconds, and each rank draws its own inputs.
"""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from self_referential_weight_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 1.5 + rank          # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(local)
        wl = bench.rank_workload(inputs.workload("tiny"), rank)
        x, _ = inputs.make_inputs(wl)
        out[world + rank] = float(x.sum())
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_per_rank_inputs():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Array("d", 2 * world)
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    vals = list(out)
    assert vals[0] == vals[1] == 2.5            # every rank sees the slowest rank's time
    assert vals[2] != vals[3]                   # ranks draw different inputs


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25


def test_rank_zero_keeps_the_named_workload():
    wl = inputs.workload("mid")
    assert bench.rank_workload(wl, 0) is wl
    assert bench.rank_workload(wl, 3).seed == wl.seed + 3000
    assert np.isclose(bench.rank_workload(wl, 3).head_tokens, wl.head_tokens)
