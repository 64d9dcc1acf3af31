"""The data-parallel bookkeeping of bench.py with two ranks on the CPU (gloo):
per-rank token batches differ, every rank sees the slowest rank's time, and
the whole-job value counts every rank's bytes.  The path itself has no
cross-rank exchange, so nothing else travels between ranks."""
from __future__ import annotations

import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from unpermute_routing_indices_gb300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed = bench.rank_seed(wl.ROUTED["tiny"]["seed"], rank)
        idx, _, _ = wl.routing("tiny", seed=seed)
        local_ms = 1.0 + 2.0 * rank                 # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        dist.barrier()
        out[rank] = (ms, int(idx.sum()), bench.job_throughput(10**9, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_the_slowest_time_and_sum_their_bytes():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    (ms0, s0, v0), (ms1, s1, v1) = out[0], out[1]
    assert ms0 == ms1 == 3.0
    assert s0 != s1                                  # independent batches
    assert v0 == v1 == bench.job_throughput(10**9, 2, 3.0)
    np.testing.assert_allclose(v0, 2 * 1e9 / 3e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.rank_seed(1003, 0) == 1003


def test_map_launch_count():
    """The kernels mp_build_map launches, as the bench counts them: one CTA or
    one cluster up to 32,768 routes; count + rank beyond; + scan when the
    count matrix passes 32,768 entries."""
    assert bench.map_launches(512, 128) == 1
    assert bench.map_launches(32768, 128) == 1
    assert bench.map_launches(32769, 128) == 2
    assert bench.map_launches(131072, 128) == 2       # the skewed step: 64 tiles
    assert bench.map_launches(262144, 256) == 2       # large: 64 tiles of 4,096
    assert bench.map_launches(131072, 1024) == 3      # 1,025 x 64 counts
