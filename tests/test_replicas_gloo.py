"""The multi-GPU path of the benchmark, on the CPU with two gloo ranks.

The decode path does not shard within a step: N GPUs run N independent
replicas (weak scaling), and the job's time is the slowest rank's.  This test
runs the benchmark's own reduction helpers in two processes over gloo.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        own = 10.0 + 5.0 * rank            # rank 1 is the slower replica
        job = bench.slowest_rank_ms(own)
        results[rank] = (job, bench.replica_tokens_per_s(job / 4, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a process that already runs torch threads
        results = m.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        got = dict(results)
    assert got[0][0] == got[1][0] == 15.0               # max over ranks, seen by every rank
    assert got[0][1] == pytest.approx(2 * 1000.0 / (15.0 / 4))


def test_single_process_returns_its_own_time():
    import bench
    assert not dist.is_initialized()
    assert bench.slowest_rank_ms(3.25) == 3.25
    assert bench.replica_tokens_per_s(2.0, 1) == 500.0
