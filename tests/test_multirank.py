"""The multi-process host logic of the bench, on CPU with the gloo backend
(world size 2): each rank runs an independent replica (the path has no
exchange step), the job's time per step is the slowest rank's, and the
whole-job throughput counts every replica's tokens over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.5, 2.25][rank]                        # the second replica is slower
    slowest = bench.max_over_ranks(ms, world, "cpu")
    out[rank] = (slowest, bench.job_tokens_per_s(8192, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for rank in range(world):
        slowest, tps = out[rank]
        assert slowest == 2.25
        assert tps == pytest.approx(8192 * 2 / 2.25e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.job_tokens_per_s(100, 1, 2.0) == pytest.approx(5e4)
