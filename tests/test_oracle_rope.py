"""Pins for the oracle rotary embedding (CPU only): closed forms of a single
rotation, RoPE's relative-position property, norm preservation, untouched
channels, and the window-local position rule (restart per window, text
offset on the t axis)."""
import math

import numpy as np

from oracle import plan as op
from oracle import rope as orp


def test_single_pair_closed_form():
    x = np.zeros((1, 1, 128)); x[0, 0, 0] = 1.0        # pair 0 of the t block
    y = orp.rope(x, np.array([[3.0, 0.0, 0.0]]))
    assert abs(y[0, 0, 0] - math.cos(3.0)) < 1e-15 and abs(y[0, 0, 1] - math.sin(3.0)) < 1e-15
    x = np.zeros((1, 1, 128)); x[0, 0, 42 + 2 * 5 + 1] = 2.0   # pair 5 of the h block, odd channel
    y = orp.rope(x, np.array([[0.0, 7.0, 0.0]]))
    ang = 7.0 * 10000.0 ** (-10.0 / 42)
    assert abs(y[0, 0, 52] + 2.0 * math.sin(ang)) < 1e-14 and abs(y[0, 0, 53] - 2.0 * math.cos(ang)) < 1e-14


def test_relative_position_property_norms_and_tail():
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal((2, 1, 3, 128))
    p, p2, shift = np.array([[5.0, 2.0, 9.0]]), np.array([[1.0, 4.0, 3.0]]), np.array([[11.0, -3.0, 6.0]])
    dot = lambda a, b: np.einsum("nhd,nhd->nh", a, b)
    # q.k after rotation depends only on the position difference
    assert np.allclose(dot(orp.rope(q, p), orp.rope(k, p2)),
                       dot(orp.rope(q, p + shift), orp.rope(k, p2 + shift)), atol=1e-12)
    y = orp.rope(q, p)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(q, axis=-1), atol=1e-12)
    assert np.array_equal(y[..., 126:], q[..., 126:])
    assert np.array_equal(orp.rope(q, np.zeros((1, 3))), q)


def test_positions_restart_per_window_and_offset_text():
    grid, L = (4, 10, 12, 2, 2, 2), 5
    pv, pt = orp.positions(*grid, op.SHIFTED, L)
    off, ids = op.layout_tables(*grid, op.SHIFTED)
    T, H, W = grid[:3]
    boxes = op.layout_boxes(*grid, op.SHIFTED)
    for wdx, ((t0, _), (h0, _), (w0, _)) in enumerate(boxes):
        first = off[wdx]
        assert tuple(pv[first]) == (L, 0, 0)                # every window restarts at (text_len, 0, 0)
        for r in range(off[wdx], off[wdx + 1]):
            c = ids[r]
            t, h, w = c // (H * W), (c // W) % H, c % W
            assert tuple(pv[r]) == (L + t - t0, h - h0, w - w0)
    assert pt.tolist() == [[l, l, l] for l in range(L)]
