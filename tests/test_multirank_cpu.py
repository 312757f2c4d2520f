"""The N>1 bench path on CPU: two gloo ranks aggregate their step times by max
and report the whole-job rate (weak scaling, one replica per rank)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank)          # rank 1 is the slow one
    rate = bench.whole_job_tokens_per_s(8, world, ms)
    dist.barrier()
    out[rank] = (ms, rate)
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 2.0
    assert out[0][1] == pytest.approx(2 * 8 / 2e-3)


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(8, 1, 4.0) == pytest.approx(2000.0)
