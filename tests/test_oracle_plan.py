"""Pins for the oracle's window geometry and re-layout (CPU only).

Each check ties oracle.plan / oracle.permute to something other than the
oracle itself: hand-derived values of the page's formula (tests/golden), the
page's invariants (exact partition, ids = windowed arange, window count grows
but window size does not), and brute force on small grids.
"""
import itertools
import random

import numpy as np
import pytest

from oracle import plan as op
from oracle import permute as opm


def test_window_size_golden(golden):
    rows = golden("window_sizes.txt")
    assert len(rows) >= 10
    for r in rows:
        T, H, W, nt, nh, nw, wt, wh, ww = map(int, r)
        assert op.window_size(T, H, W, nt, nh, nw) == (wt, wh, ww), r


def _parse_intervals(fields):
    return [tuple(map(int, f.split(":"))) for f in fields]


def test_intervals_golden(golden):
    rows = golden("intervals.txt")
    for r in rows:
        kind, n, w = r[0], int(r[1]), int(r[2])
        fn = {"regular": op.regular_intervals, "shifted": op.shifted_intervals,
              "shifted_ceil": lambda n, w: op.shifted_intervals(n, w, half="ceil")}[kind]
        assert fn(n, w) == _parse_intervals(r[3:]), r
    assert {r[0] for r in rows} == {"regular", "shifted", "shifted_ceil"}


def _layout(name):
    return {"regular": op.REGULAR, "shifted": op.SHIFTED}[name]


def test_window_counts_golden(golden):
    for r in golden("window_counts.txt"):
        T, H, W, nt, nh, nw = map(int, r[:6])
        off, ids = op.layout_tables(T, H, W, nt, nh, nw, _layout(r[6]))
        sizes = np.diff(off)
        assert (len(sizes), sizes.min(), sizes.max()) == tuple(map(int, r[7:10])), r


def test_window_tokens_pr1_golden(golden):
    for r in golden("window_tokens_pr1.txt"):
        off, _ = op.layout_tables(2, 45, 80, 1, 3, 3, _layout(r[0]))
        assert np.diff(off).tolist() == list(map(int, r[1:])), r


def _brute_force_ids(T, H, W, nt, nh, nw, layout, half="floor"):
    """Layout order from scratch: for every token find the window that holds
    it by scanning the per-axis intervals, then order tokens by
    (window index in w->h->t enumeration, canonical id).  Within a box,
    row-major (t,h,w) order is increasing canonical id."""
    wt, wh, ww = op.window_size(T, H, W, nt, nh, nw)
    if layout == op.REGULAR:
        ax = op.regular_intervals
    else:
        ax = lambda n, w: op.shifted_intervals(n, w, half)
    ti, hi, wi = ax(T, wt), ax(H, wh), ax(W, ww)

    def find(ints, x):
        hits = [i for i, (a, b) in enumerate(ints) if a <= x < b]
        assert len(hits) == 1  # exact partition of the axis
        return hits[0]

    key = []
    for t in range(T):
        for h in range(H):
            for w in range(W):
                win = (find(wi, w) * len(hi) + find(hi, h)) * len(ti) + find(ti, t)
                key.append((win, (t * H + h) * W + w))
    key.sort()
    return np.asarray([cid for _, cid in key], dtype=np.int64)


SMALL_GRIDS = [
    (2, 45, 80, 1, 3, 3),
    (5, 9, 16, 2, 1, 1),
    (3, 7, 11, 2, 2, 3),
    (7, 12, 5, 3, 2, 2),
    (1, 1, 1, 1, 1, 1),
    (4, 10, 10, 1, 4, 4),
    (33, 6, 4, 4, 1, 2),   # T > 30
]


@pytest.mark.parametrize("grid", SMALL_GRIDS)
@pytest.mark.parametrize("layout,half", [(op.REGULAR, "floor"), (op.SHIFTED, "floor"), (op.SHIFTED, "ceil")])
def test_ids_match_brute_force(grid, layout, half):
    off, ids = op.layout_tables(*grid, layout, half=half)
    assert np.array_equal(ids, _brute_force_ids(*grid, layout, half))
    assert off[0] == 0 and off[-1] == ids.size


def _random_grids(n, seed=7):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        out.append((rng.randint(1, 40), rng.randint(1, 70), rng.randint(1, 130),
                    rng.randint(1, 5), rng.randint(1, 4), rng.randint(1, 4)))
    return out


@pytest.mark.parametrize("grid", _random_grids(40) + [(21, 45, 80, 4, 3, 3),
                                                      (21, 68, 120, 4, 3, 3),
                                                      (30, 90, 160, 4, 3, 3)])
def test_layouts_partition_the_grid(grid):
    """§Window layouts: both methods produce an exact partition."""
    T, H, W = grid[:3]
    wt, wh, ww = op.window_size(*grid)
    if min(wt, wh, ww) <= 0:
        pytest.skip("window of size 0 (rejected by the planner)")
    for layout, half in ((op.REGULAR, "floor"), (op.SHIFTED, "floor"), (op.SHIFTED, "ceil")):
        off, ids = op.layout_tables(*grid, layout, half=half)
        assert np.array_equal(np.sort(ids), np.arange(T * H * W))
        assert np.all(np.diff(off) > 0)  # no empty window


@pytest.mark.parametrize("grid", _random_grids(40, seed=11))
def test_shifted_differs_when_an_axis_has_two_windows(grid):
    """§Window layouts: the shifted layout is genuinely different."""
    T, H, W = grid[:3]
    wt, wh, ww = op.window_size(*grid)
    if min(wt, wh, ww) <= 0:
        pytest.skip("window of size 0")
    # A window of length 1 has its cuts moved by floor(1/2) = 0, so only an
    # axis with 2 <= w < n changes.
    multi = any(2 <= w < n for w, n in ((wt, T), (wh, H), (ww, W)))
    b_reg = op.layout_boxes(*grid, op.REGULAR)
    b_shf = op.layout_boxes(*grid, op.SHIFTED)
    assert (b_reg != b_shf) == multi


def test_window_count_grows_size_does_not():
    """§Motivation: a higher resolution adds windows, never window size."""
    grids = [(27, 48), (36, 64), (45, 80), (54, 96), (68, 120), (72, 128),
             (90, 160), (108, 192), (135, 240)]
    counts = []
    for H, W in grids:
        assert op.window_size(21, H, W, 4, 3, 3) == (6, 15, 27)
        counts.append(len(op.layout_boxes(21, H, W, 4, 3, 3, op.REGULAR)))
    assert counts == sorted(counts) and counts[-1] > counts[0]


def test_canonical_layout_is_identity():
    off, ids = op.layout_tables(3, 4, 5, 1, 1, 1, op.CANONICAL)
    assert off.tolist() == [0, 60] and np.array_equal(ids, np.arange(60))


def test_canonical_id_formula():
    """§Window layouts: canonical id of (t,h,w) is (t*H+h)*W+w.  Windowing
    arange must give exactly that id for the first token of every box."""
    T, H, W = 7, 12, 5
    off, ids = op.layout_tables(T, H, W, 3, 2, 2, op.SHIFTED)
    boxes = op.layout_boxes(T, H, W, 3, 2, 2, op.SHIFTED)
    for k, ((t0, _), (h0, _), (w0, _)) in enumerate(boxes):
        assert ids[off[k]] == (t0 * H + h0) * W + w0


# ---------------------------------------------------------------- permute --

def _ids(grid, layout):
    return op.layout_tables(*grid, layout)[1]


@pytest.mark.parametrize("grid", SMALL_GRIDS[:4] + [(21, 45, 80, 4, 3, 3)])
def test_permute_moves_each_token_to_its_row(grid):
    """Rows tagged with their canonical id must land where ids_dst says."""
    layouts = (op.CANONICAL, op.REGULAR, op.SHIFTED)
    for a, b in itertools.permutations(layouts, 2):
        ia, ib = _ids(grid, a), _ids(grid, b)
        src = np.stack([ia, -ia], axis=1)          # row p carries id ia[p]
        dst = opm.permute_rows(src, ia, ib)
        assert np.array_equal(dst[:, 0], ib) and np.array_equal(dst[:, 1], -ib)


def test_permute_round_trip_and_composition():
    grid = (5, 9, 16, 2, 1, 1)
    rng = np.random.default_rng(0)
    ic, ir, isf = (_ids(grid, l) for l in (op.CANONICAL, op.REGULAR, op.SHIFTED))
    x = rng.standard_normal((ic.size, 6)).astype(np.float32)
    xr = opm.permute_rows(x, ic, ir)
    assert np.array_equal(opm.permute_rows(opm.permute_rows(xr, ir, isf), isf, ir), xr)
    direct = opm.permute_rows(xr, ir, isf)
    via_c = opm.permute_rows(opm.permute_rows(xr, ir, ic), ic, isf)
    assert np.array_equal(direct, via_c)
    assert np.array_equal(opm.permute_rows(xr, ir, ic), x)
