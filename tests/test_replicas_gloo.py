"""The multi-rank (replicas-only) path of bench.py on CPU: two gloo ranks time
different amounts, the job's time is the slowest rank's, and the whole-job
throughput counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    r, w = bench.dist()
    assert (r, w) == (rank, world)
    ms_rank = 2.0 + 3.0 * rank  # rank 1 is the slow one
    value, ms = bench.job_throughput(1e9, ms_rank, w)
    bench.barrier(w)
    out[rank] = (value, ms)
    torch.distributed.destroy_process_group()


def test_two_replicas_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for rank in range(world):
        value, ms = out[rank]
        assert ms == pytest.approx(5.0)               # the slowest rank
        assert value == pytest.approx(2e9 / 5e-3)     # both ranks' units over that time
