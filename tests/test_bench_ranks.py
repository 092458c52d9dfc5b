"""Host logic of the multi-GPU form (independent replicas, one process per
GPU): the whole-job throughput takes the slowest rank's time over a real
world-size-2 process group (gloo on CPU; the GPU runs use NCCL)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r timed its steps in 100 + 50 r ms and processed 1000 tokens
    ms, value = bench.reduce_timing(100.0 + 50.0 * rank, 1000, world)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_uses_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == 150.0
        assert value == pytest.approx(2000 / 0.150)


def test_single_process_needs_no_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_timing(200.0, 512, 1) == (200.0, pytest.approx(512 / 0.2))
