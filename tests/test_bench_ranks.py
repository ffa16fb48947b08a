"""bench.py's multi-rank bookkeeping, on CPU: world size 2 over gloo.

The layer's units are independent sequences, so N GPUs run N replicas of the
per-GPU work with no collective on the data path; the only collectives are the
bench's barrier and the maximum of the ranks' times, and the reported rate
counts the units of every rank over the slowest rank's time.
"""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out) -> None:
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.rank_max(1.0 + 0.5 * rank, world, "cpu")  # the last rank is the slowest
        dist.barrier()
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, _free_port(), out), nprocs=2, join=True)
        assert dict(out) == {0: 1.5, 1: 1.5}


def test_single_rank_needs_no_process_group():
    assert bench.rank_max(0.7, 1, "cpu") == 0.7


def test_job_rate_counts_the_units_of_every_rank():
    assert bench.job_rate(65536, 1, 1.0) == 65536 * 1e3
    # four replicas of 65536 tokens in 2 ms (the slowest rank's time)
    assert abs(bench.job_rate(65536, 4, 2.0) - 65536 * 4 / 2e-3) < 1e-6
