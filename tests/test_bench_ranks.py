"""The benchmark's multi-GPU aggregation (independent replicas, one process
per GPU) on CPU: two gloo ranks with different step times must agree on the
slowest rank's time and on the whole-job throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [812.5, 1234.0][rank]                     # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, "cpu")
    out[rank] = (worst, bench.job_throughput(worst, 4096, 1, world), bench.job_throughput(worst, 64, 16, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1]
    worst, tput1, tput16 = out[0]
    assert worst == 1234.0
    assert tput1 == pytest.approx(2 * 4096 / 1.234)
    assert tput16 == pytest.approx(2 * 64 * 16 / 1.234)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_throughput(1000.0, 10, 2, 1) == pytest.approx(20.0)
