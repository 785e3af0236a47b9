"""bench.py's multi-rank bookkeeping on CPU with two gloo ranks: the job's
time is the slowest rank's and its throughput counts every rank's bytes.
(The decode path itself has no exchange step; ranks are replicas.)"""

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_setup() == (world, rank, rank)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")  # rank 1 is slower
        out[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: 15.0, 1: 15.0}
    # 2 ranks x 1e9 bytes in 2 ms -> 1000 GB/s
    assert abs(bench.job_throughput(1e9, 2, 2.0) - 1000.0) < 1e-9


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5
