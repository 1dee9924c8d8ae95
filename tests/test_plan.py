"""The C++ planner (arithmetic) equals the oracle planner (windowing an arange
cube) bit for bit: offsets, id tables and boxes (CPU only)."""
import random

import numpy as np
import pytest

from oracle import plan as op


@pytest.fixture(scope="module")
def wp():
    import __graft_entry__
    __graft_entry__.build()
    from video_dit_shifted_gb300 import wp as _wp
    return _wp


SWEEP = [(T, H, W, 4, 3, 3) for (H, W) in ((45, 80), (68, 120), (90, 160)) for T in (5, 21, 30)]
CONFIGS = [(2, 45, 80, 1, 3, 3), (21, 45, 80, 4, 3, 3), (21, 68, 120, 4, 3, 3), (30, 90, 160, 4, 3, 3)]


def _random_grids(n, seed=3):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        g = (rng.randint(1, 45), rng.randint(1, 80), rng.randint(1, 140),
             rng.randint(1, 6), rng.randint(1, 5), rng.randint(1, 5))
        if min(op.window_size(*g)) >= 1:
            out.append(g)
    return out


@pytest.mark.parametrize("grid", sorted(set(SWEEP + CONFIGS)) + _random_grids(120))
def test_tables_match_oracle(wp, grid):
    plan = wp.Plan(*grid)
    for layout in (op.CANONICAL, op.REGULAR, op.SHIFTED):
        off, ids, boxes = plan.host_tables(layout)
        o_off, o_ids = op.layout_tables(*grid, layout)
        assert np.array_equal(off.astype(np.int64), o_off), (grid, layout)
        assert np.array_equal(ids.astype(np.int64), o_ids), (grid, layout)
        o_boxes = np.array([[*t, *h, *w] for t, h, w in op.layout_boxes(*grid, layout)])
        assert np.array_equal(boxes, o_boxes), (grid, layout)
        info = plan.info(layout)
        assert info["nwin"] == len(o_off) - 1
        assert info["max_tokens"] == int(np.diff(o_off).max())
        assert info["window"] == op.window_size(*grid)
    plan.close()


def test_window_size_matches_oracle_widely(wp):
    rng = random.Random(5)
    for _ in range(2000):
        g = (rng.randint(1, 100), rng.randint(1, 400), rng.randint(1, 400),
             rng.randint(1, 8), rng.randint(1, 8), rng.randint(1, 8))
        want = op.window_size(*g)
        if min(want) < 1:
            continue
        plan = wp.Plan(*g) if g[0] * g[1] * g[2] <= 200000 else None
        if plan is None:
            continue
        assert plan.info(op.REGULAR)["window"] == want, g
        plan.close()
