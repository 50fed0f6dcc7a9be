"""Multi-replica bookkeeping of bench.py on two gloo ranks (CPU): the timed
region is the slowest rank's, the throughput counts every rank's work."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, store_file, out):
    # a file rendezvous: no port to race for with other processes on the machine
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="file://" + store_file, rank=rank,
                            world_size=world)
    import bench
    local_ms = [12.0, 20.0][rank]
    ms, value = bench.job_throughput(local_ms, world, 3.0e12, 5, torch.device("cpu"))
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_throughput_uses_max_time_and_all_work(tmp_path):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    store_file = str(tmp_path / "rendezvous")
    mp.start_processes(_worker, args=(world, store_file, out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 20.0
        assert value == pytest.approx(world * 3.0e12 * 5 / 0.020 / 1e12)


def test_single_rank_throughput():
    import bench
    ms, value = bench.job_throughput(10.0, 1, 2.0e12, 4, torch.device("cpu"))
    assert ms == 10.0 and value == pytest.approx(2.0e12 * 4 / 0.010 / 1e12)
