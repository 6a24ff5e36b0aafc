"""The multi-GPU path of the benchmark is replicas only (every sequence and
head is independent, no collective on the data path): the whole-job value is
the units of all ranks over the slowest rank's time.  Checked here with two
gloo ranks on CPU (the timing reduction is the only collective)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_total = [100.0, 130.0][rank]          # rank 1 is the slow one
    ms_step, value = bench.replica_throughput(ms_total, 10, 5e12, world, dist, torch.device("cpu"))
    out[rank] = (ms_step, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms_step, value = res[r]
        assert ms_step == 13.0                     # MAX over ranks, per step
        assert abs(value - 2 * 5e12 / 13e-3 / 1e12) < 1e-9


def test_single_replica_needs_no_collective():
    ms_step, value = bench.replica_throughput(50.0, 5, 1e12, 1)
    assert ms_step == 10.0 and abs(value - 1e12 / 10e-3 / 1e12) < 1e-12
