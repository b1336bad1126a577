"""bench.py's multi-process path on CPU: two gloo ranks, each timing its own
replica, agree on the slowest rank's time; whole-job throughput counts every
rank's units; the reference arm does no work on ranks other than 0."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 5.0 - rank]  # rank 1 is slower in the first timing only
    got = bench.max_over_ranks(mine, dist)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == [11.0, 5.0]


def test_job_throughput_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(1000, 2, 500.0) == pytest.approx(4000.0)
    assert bench.max_over_ranks([1.5, 2.5], None) == [1.5, 2.5]


def test_reference_arm_does_nothing_on_other_ranks(capsys):
    sys.path.insert(0, ROOT)
    import bench
    bench.run_reference(None, rank=1, world=2)  # must return before touching args
    assert capsys.readouterr().out == ""
