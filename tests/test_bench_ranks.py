"""bench.py's multi-replica bookkeeping on two CPU processes (gloo): the
barrier and the max over ranks of the step time."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"], os.environ["MASTER_PORT"] = "127.0.0.1", str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(dist)
    out[rank] = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, torch.device("cpu"))
    dist.destroy_process_group()


def test_max_over_two_ranks():
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}
