"""Pins for the oracle multi-device planner (CPU only): hand-derived LPT
examples (tests/golden/lpt_example.txt), LPT invariants, and a simulated
all-to-all that must leave every rank holding exactly its destination rows."""
import numpy as np
import pytest

from oracle import plan as op
from oracle import ranks as ork


def test_lpt_golden(golden):
    for r in golden("lpt_example.txt"):
        parts = " ".join(r).split("|")
        world = int(parts[0])
        sizes = list(map(int, parts[1].split()))
        want_rank = list(map(int, parts[2].split()))
        want_load = list(map(int, parts[3].split()))
        assert ork.lpt_assign(sizes, world) == (want_rank, want_load)


@pytest.mark.parametrize("grid", [(21, 68, 120, 4, 3, 3), (30, 90, 160, 4, 3, 3)])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_lpt_balance_bound(grid, world):
    """Greedy on sorted sizes: loads differ by at most the largest window."""
    for layout in (op.REGULAR, op.SHIFTED):
        off, _ = op.layout_tables(*grid, layout)
        sizes = np.diff(off)
        wr, load = ork.lpt_assign(sizes, world)
        assert sum(load) == sizes.sum()
        assert max(load) - min(load) <= sizes.max()
        for r in range(world):
            assert load[r] == sizes[np.array(wr) == r].sum()


def _simulate(grid, world, a, b):
    src = op.layout_tables(*grid, a)
    dst = op.layout_tables(*grid, b)
    C, req, send, recv = ork.exchange(src, dst, world)
    ws, _ = ork.lpt_assign(np.diff(src[0]), world)
    wd, _ = ork.lpt_assign(np.diff(dst[0]), world)
    held = [np.array(ork.rank_tokens(*src, ws, r)) for r in range(world)]  # rows = canonical ids
    for d in range(world):
        # all_to_all: rank d receives, from r = 0..world-1, r's segment for d
        segs = []
        for r in range(world):
            start = int(C[r, :d].sum())
            segs.append(held[r][send[r]][start:start + int(C[r, d])])
        got = np.concatenate(segs) if segs else np.zeros(0, np.int64)
        local = got[np.argsort(recv[d], kind="stable")]
        assert np.array_equal(local, np.array(ork.rank_tokens(*dst, wd, d)))
        assert C[:, d].sum() == len(ork.rank_tokens(*dst, wd, d))
    return C, req


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_exchange_delivers_every_row(world):
    grid = (5, 45, 80, 4, 3, 3)
    for a, b in [(op.REGULAR, op.SHIFTED), (op.SHIFTED, op.REGULAR), (op.CANONICAL, op.REGULAR)]:
        C, req = _simulate(grid, world, a, b)
        if world == 1:
            assert C.tolist() == [[grid[0] * grid[1] * grid[2]]] and not req


def test_same_layout_needs_no_exchange():
    grid = (5, 45, 80, 4, 3, 3)
    C, req = _simulate(grid, 4, op.REGULAR, op.REGULAR)
    assert not req and np.count_nonzero(C - np.diag(np.diag(C))) == 0
