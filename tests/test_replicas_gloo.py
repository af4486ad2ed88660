"""The multi-GPU path of bench.py is "replicas only": every rank runs its own
SGEMM, and the only cross-rank step is the max-over-ranks of the step time.
That reduction and the whole-job throughput are checked here with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world, device="cpu")
        out[rank] = (slowest, bench.replica_throughput(2.0e9, slowest, world))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_throughput_two_gloo_ranks():
    world = 2
    times = [2.0, 3.5]                    # ms per step on each rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        slowest, gflops = res[r]
        assert slowest == 3.5
        # 2 ranks x 2 GFLOP each in 3.5 ms
        assert gflops == pytest.approx(2 * 2.0e9 / 3.5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.replica_throughput(1e9, 1.0, 1) == pytest.approx(1000.0)
