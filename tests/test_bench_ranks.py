"""The multi-rank bench path on CPU: two gloo ranks, different step times.

bench.py under torchrun runs one independent mesh per GPU (weak scaling, no
data-path collective); the only cross-rank step is the timing: the slowest
rank's elapsed time, and the bytes of all ranks per second.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [400.0, 1000.0][rank]
        q.put((rank, bench.aggregate_ranks(dist, torch, elapsed, 2e9, 10)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        ms, world, gbs = out[rank]
        assert ms == 1000.0 and world == 2
        assert gbs == pytest.approx(2e9 * 2 * 10 / 1.0 / 1e9)


def test_single_process_needs_no_process_group():
    ms, world, gbs = bench.aggregate_ranks(None, torch, 250.0, 1e9, 4)
    assert (ms, world) == (250.0, 1) and gbs == pytest.approx(16.0)
