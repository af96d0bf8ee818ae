"""The multi-GPU path of bench.py on the CPU with the gloo backend: every rank
runs its own layer replica on its own tokens (no collective on the data path),
the job's time is the slowest rank's and its throughput counts every rank's
tokens.  world_size 2, no GPU."""
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


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(times[rank], world)
        tput = bench.job_throughput(64, world, m)
        dist.barrier()
        out[rank] = (m, tput)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(1.5, 2.0), (3.0, 0.25)])
def test_two_ranks_take_the_slowest_rank_and_count_all_tokens(times):
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, tput = res[r]
        assert m == max(times)
        assert tput == pytest.approx(world * 64 / max(times))


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.7, 1) == 0.7
    assert bench.job_throughput(16, 1, 0.5) == 32.0
