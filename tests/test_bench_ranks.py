"""The multi-rank reduction of bench.py on CPU: two gloo ranks, each with its
own replica's time and bytes; the whole-job line takes the slowest rank's
time and the sum of the bytes."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]
    e2e = [1.0, 0.75][rank]
    res = bench.combine_ranks(ms, e2e, 1000 * (rank + 1), 10 * (rank + 1), world, "cpu")
    out[rank] = res
    dist.destroy_process_group()


def test_two_ranks_take_max_time_and_summed_bytes():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    for r in (0, 1):
        assert out[r] == (12.5, 1.0, 3000.0, 30.0)


def test_one_rank_passes_through():
    import bench
    assert bench.combine_ranks(3.0, 2.0, 5, 7, 1, "cpu") == (3.0, 2.0, 5.0, 7.0)
