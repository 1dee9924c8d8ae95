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


@pytest.mark.parametrize("grid", sorted(set(SWEEP + CONFIGS)) + _random_grids(60, seed=9))
def test_half_ceil_tables_match_oracle(wp, grid):
    """The other reading of an odd half window (WP_PLAN_HALF_CEIL) against the
    oracle's half="ceil": shifted tables bit for bit; regular and canonical
    tables, and every layout of a grid whose window sizes are all even, the
    same as the default plan's."""
    plan = wp.Plan(*grid, half="ceil")
    base = wp.Plan(*grid)
    for layout in (op.CANONICAL, op.REGULAR, op.SHIFTED):
        off, ids, boxes = plan.host_tables(layout)
        o_off, o_ids = op.layout_tables(*grid, layout, half="ceil")
        assert np.array_equal(off.astype(np.int64), o_off), (grid, layout)
        assert np.array_equal(ids.astype(np.int64), o_ids), (grid, layout)
        o_boxes = np.array([[*t, *h, *w] for t, h, w in op.layout_boxes(*grid, layout, half="ceil")])
        assert np.array_equal(boxes, o_boxes), (grid, layout)
        b_off, b_ids, _ = base.host_tables(layout)
        same = layout != op.SHIFTED or all(w % 2 == 0 or w >= n for w, n in zip(op.window_size(*grid), grid[:3]))
        if same:
            assert np.array_equal(off, b_off) and np.array_equal(ids, b_ids), (grid, layout)
    plan.close()
    base.close()


def test_half_ceil_removes_the_one_row_slices(wp):
    """1080p-like grid (T, H, W = 21, 68, 120; window 6 x 15 x 27): the floor
    reading cuts h at 7, 22, 37, 52, 67 (a 1-row slice 67:68) and w at 13,
    40, 67, 94, so its smallest window is 3 x 1 x 13 = 39 tokens; the ceil
    reading cuts h at 8, 23, 38, 53 and w at 14, 41, 68, 95 (t, w = 6: 3, 9,
    15 either way), smallest window 3 x 8 x 14 = 336.  Derived by hand."""
    grid = (21, 68, 120, 4, 3, 3)
    for half, smallest in (("floor", 39), ("ceil", 336)):
        plan = wp.Plan(*grid, half=half)
        assert plan.info(op.SHIFTED)["nwin"] == len(op.layout_boxes(*grid, op.SHIFTED, half=half))
        off, _, boxes = plan.host_tables(op.SHIFTED)
        assert int(np.diff(off).min()) == smallest, half
        assert (int((boxes[:, 3] - boxes[:, 2]).min()) == 1) == (half == "floor")
        plan.close()


def test_plan_flags_are_checked(wp):
    import ctypes
    h = ctypes.c_void_p()
    assert wp.lib().wp_plan_create_ex(2, 45, 80, 1, 3, 3, 2, ctypes.byref(h)) == 1      # WP_EINVAL
    assert "flags" in wp.lib().wp_last_error().decode()
    with pytest.raises(ValueError):
        wp.Plan(2, 45, 80, 1, 3, 3, half="round")


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
