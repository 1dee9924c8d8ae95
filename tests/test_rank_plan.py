"""The C++ multi-device planner against the oracle (CPU only), and a real
two-process all-to-all over gloo that moves rows with the planner's tables."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import plan as op
from oracle import ranks as ork


@pytest.fixture(scope="module")
def wp():
    import __graft_entry__
    __graft_entry__.build()
    from video_dit_shifted_gb300 import wp as _wp
    return _wp


@pytest.mark.parametrize("grid", [(21, 68, 120, 4, 3, 3), (5, 45, 80, 4, 3, 3), (3, 7, 11, 2, 2, 3)])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_assign_matches_oracle(wp, grid, world):
    plan = wp.Plan(*grid)
    for layout in (op.CANONICAL, op.REGULAR, op.SHIFTED):
        wr, load = plan.assign(layout, world)
        o_wr, o_load = ork.lpt_assign(np.diff(op.layout_tables(*grid, layout)[0]), world)
        assert wr.tolist() == o_wr and load.tolist() == o_load
    plan.close()


@pytest.mark.parametrize("world", [1, 2, 4])
def test_exchange_matches_oracle(wp, world):
    grid = (5, 45, 80, 4, 3, 3)
    plan = wp.Plan(*grid)
    for a, b in [(op.REGULAR, op.SHIFTED), (op.SHIFTED, op.REGULAR), (op.CANONICAL, op.SHIFTED)]:
        C, req, send, recv = ork.exchange(op.layout_tables(*grid, a), op.layout_tables(*grid, b), world)
        for r in range(world):
            c2, req2, s2, r2 = plan.exchange(a, b, world, r)
            assert np.array_equal(c2, C) and req2 == req
            assert s2.tolist() == send[r] and r2.tolist() == recv[r]
    plan.close()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, grid, a, b, out):
    os.environ["MASTER_ADDR"], os.environ["MASTER_PORT"] = "127.0.0.1", str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import __graft_entry__
    __graft_entry__.build()
    from video_dit_shifted_gb300 import wp
    plan = wp.Plan(*grid)
    C, req, send, recv = plan.exchange(a, b, world, rank)
    # rows this rank holds in layout a (local order), tagged by canonical id
    win_off, ids, _ = plan.host_tables(a)
    wr, _ = plan.assign(a, world)
    mine = np.concatenate([ids[win_off[w]:win_off[w + 1]] for w in range(len(wr)) if wr[w] == rank]
                          or [np.zeros(0, np.int32)])
    x = torch.from_numpy(np.stack([mine, -mine], 1).astype(np.int64))
    inp = x[torch.from_numpy(send.astype(np.int64))]
    outp = torch.empty((int(C[:, rank].sum()), 2), dtype=torch.int64)
    if req:  # §Plan A: every rank takes the same branch, decided from C
        dist.all_to_all_single(outp, inp, [int(v) for v in C[:, rank]], [int(v) for v in C[rank]])
    else:
        outp.copy_(inp)
    local = torch.empty_like(outp)
    local[torch.from_numpy(recv.astype(np.int64))] = outp
    d_off, d_ids, _ = plan.host_tables(b)
    wd, _ = plan.assign(b, world)
    want = np.concatenate([d_ids[d_off[w]:d_off[w + 1]] for w in range(len(wd)) if wd[w] == rank]
                          or [np.zeros(0, np.int32)])
    out[rank] = int(np.array_equal(local[:, 0].numpy(), want) and np.array_equal(local[:, 1].numpy(), -want))
    plan.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("a,b", [(op.REGULAR, op.SHIFTED), (op.SHIFTED, op.REGULAR)])
def test_gloo_two_rank_exchange(wp, a, b):
    """Two CPU processes exchange rows with all_to_all_single using the
    planner's split sizes, send order and receive positions; each must end
    holding exactly its destination rows in its local order."""
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), (5, 45, 80, 4, 3, 3), a, b, out),
                       nprocs=world, join=True, start_method="spawn")
    assert dict(out) == {0: 1, 1: 1}
