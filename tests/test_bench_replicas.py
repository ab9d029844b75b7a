"""The multi-GPU path of bench.py (replicas: one process per GPU, no data-path collective),
run as two gloo ranks on CPU: the slowest rank's time reaches every rank, the whole-job
throughput counts every rank's queries, and the launch environment is read as torchrun
sets it."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        secs = bench.max_over_ranks(1.0 + rank, torch.device("cpu"), ws)
        value = bench.replica_throughput(1000, 10, secs, ws)
        out[rank] = torch.tensor([ws, r, local, secs, value], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank_and_count_every_rank(world):
    out = torch.zeros((world, 5), dtype=torch.float64).share_memory_()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ws, r, local, secs, value = out[rank].tolist()
        assert (ws, r, local) == (world, rank, rank)
        assert secs == float(world)                     # rank world-1 took 1 + (world-1) s
        assert value == world * 1000 * 10 / float(world)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(2.5, torch.device("cpu"), 1) == 2.5
    assert bench.replica_throughput(100, 4, 2.0, 1) == 200.0
