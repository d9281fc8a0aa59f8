"""The multi-GPU path of bench.py, on CPU: the layer has no exchange step, so
N GPUs run N independent replicas and the job's throughput is all ranks'
work over the slowest rank's time. Two gloo ranks check that aggregation
(the same functions bench.py calls under torchrun with NCCL)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [0.25, 0.5][rank]          # rank 1 is the slow replica
    work = 1.0e12
    out[rank] = (bench.replica_max(seconds, world), bench.replica_throughput(work, seconds, world))
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_the_slowest_rank():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t_max, thr = res[r]
        assert t_max == pytest.approx(0.5)
        assert thr == pytest.approx(world * 1.0e12 / 0.5)


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_max(0.3, 1) == 0.3
    assert bench.replica_throughput(2.0, 0.5, 1) == pytest.approx(4.0)
