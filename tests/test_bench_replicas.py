"""The multi-replica aggregation of bench.py on CPU, two gloo ranks.

Each rank is an independent replica (no collective on the data path); the
job's time is the slowest rank's and its bytes are the sum over ranks."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        times = [10.0 + 5.0 * rank, 20.0 - 5.0 * rank]   # rank 1 slower in the first, faster in the second
        tmax, gbs = bench.aggregate(times, weight_bytes=1e9, world=world)
        out[rank] = (tmax, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_bytes():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        tmax, gbs = out[r]
        assert tmax == [15.0, 20.0]
        assert gbs == pytest.approx([2e9 / 15e-3 / 1e9, 2e9 / 20e-3 / 1e9])


def test_single_rank_needs_no_process_group():
    import bench
    tmax, gbs = bench.aggregate([4.0], weight_bytes=2e9, world=1)
    assert tmax == [4.0] and gbs == pytest.approx([500.0])
