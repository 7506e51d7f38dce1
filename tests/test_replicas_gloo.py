"""The N > 1 path's host logic on CPU: world-size-2 gloo process group.

The path does not shard (independent replicas, no data-path collective);
what crosses ranks is the timing: the slowest rank's time and the
whole-job rate over it.  Also: only rank 0 reports."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from weight_streaming_nf4_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = replicas.max_over_ranks(times[rank], dist, "cpu")
        rate = replicas.whole_job_rate(10.0, 3, world, t)
        out[rank] = (t, rate, replicas.is_reporter(rank))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rate_world2():
    world, port = 2, _free_port()
    times = [0.25, 0.40]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, times, out), nprocs=world, start_method="spawn")
    for r in range(world):
        t, rate, rep = out[r]
        assert t == pytest.approx(0.40)
        # two replicas of 3 steps x 10 units within the slowest rank's 0.4 s
        assert rate == pytest.approx(2 * 10.0 * 3 / 0.40)
        assert rep == (r == 0)


def test_single_process_needs_no_group():
    assert replicas.max_over_ranks(0.5) == 0.5
    assert replicas.whole_job_rate(4.0, 2, 1, 0.5) == pytest.approx(16.0)
    with pytest.raises(ValueError):
        replicas.whole_job_rate(1.0, 1, 1, 0.0)
