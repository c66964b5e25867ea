"""Host logic of the multi-GPU (replicas-only) bench path, on CPU with gloo ranks."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r reports (r+1) ms per step: the job is as slow as rank world-1
    vals = bench.max_over_ranks([rank + 1.0, 10.0 * (world - rank), 0.5], "cpu")
    q.put((rank, vals))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r] == [float(world), 10.0 * world, 0.5]


def test_job_value_is_per_step_of_the_whole_job():
    assert bench.job_value_us(2.0, 1) == 2000.0
    assert bench.job_value_us(2.0, 4) == 500.0


def test_single_process_max_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
