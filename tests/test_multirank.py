"""The N>1 path of bench.py on CPU: every rank is an independent replica (the
path has no cross-GPU step); the job time is the maximum over ranks and the
job throughput counts the work of all ranks.  Run as two gloo ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 100.0 + 25.0 * rank                  # rank 1 is the slow replica
    got = bench.max_over_ranks(mine, torch.device("cpu"))
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == 125.0
    import bench
    # whole-job throughput: both replicas' work over the slowest replica's time
    assert bench.job_tflops(2, 10, 125.0) == pytest.approx(2 * bench.STEP_FLOPS * 10 / 0.125 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
