"""Oracle window geometry (test infrastructure; see the package docstring).

Follows "Window-Aligned Sequence Parallelism (SeedVR2)", §Window layouts:

* window size is normalised to the 720p latent area 45x80:
  ``scale = sqrt(45*80/(H*W))``, ``wh = ceil(round(H*scale)/nh)``,
  ``ww = ceil(round(W*scale)/nw)``, ``wt = ceil(min(T, 30)/nt)``;
* the regular layout tiles each axis with ``[i*w, min((i+1)*w, n))``;
* the shifted layout moves every cut by half a window and clips at the axis
  ends (not a cyclic roll);
* windows are enumerated w-outermost, then h, then t innermost; tokens inside
  a window are row-major in (t, h, w);
* the canonical id of token (t, h, w) is ``(t*H + h)*W + w``, which is what one
  gets by windowing ``arange(T*H*W).reshape(T, H, W)`` -- and that is exactly
  how ``layout_tables`` builds the id table here.

Readings of points the page leaves open:

* ``round`` is Python's ``round`` on the float64 product (ties to even).
* The half-window shift of an odd window length is floored by default: cuts
  sit at ``floor((2k+1)*w/2)``; ``half="ceil"`` takes the other reading,
  ``ceil((2k+1)*w/2)``.  PARITY UNPINNED: both partition the grid, so no
  invariant on the pages distinguishes the two.
* An axis that a single window already covers (``w >= n``) has no interior cut
  to move, so its shifted interval list is the single interval ``[0, n)``.
"""
import math

import numpy as np

CANONICAL, REGULAR, SHIFTED = 0, 1, 2
LAYOUT_NAMES = {CANONICAL: "canonical", REGULAR: "regular", SHIFTED: "shifted"}
MAX_TEMPORAL_WINDOW = 30  # §Window layouts: wt is computed from min(T, 30)


def _ceil_div(a, b):
    return -(-a // b)


def window_size(T, H, W, nt, nh, nw):
    """(wt, wh, ww) from the 720p-normalised formula of §Window layouts."""
    scale = math.sqrt(45 * 80 / (H * W))
    rh = round(H * scale)
    rw = round(W * scale)
    wh = _ceil_div(rh, nh)
    ww = _ceil_div(rw, nw)
    wt = _ceil_div(min(T, MAX_TEMPORAL_WINDOW), nt)
    return wt, wh, ww


def regular_intervals(n, w):
    """[i*w, min((i+1)*w, n)) for every i that starts inside the axis."""
    return [(i * w, min((i + 1) * w, n)) for i in range(_ceil_div(n, w))]


def shifted_intervals(n, w, half="floor"):
    """Cuts moved by half a window, clipped to [0, n].  The cut after the
    k-th regular window moves to (k + 1/2) * w; for an odd w that is not an
    integer and the page does not say which way it goes: half="floor" (the
    default) takes floor, half="ceil" takes ceil."""
    if w >= n:
        return [(0, n)]
    cuts = {0, n}
    k = 0
    while True:
        num = (2 * k + 1) * w                      # the cut is num / 2
        cut = num // 2 if half == "floor" else -(-num // 2)
        if cut >= n:
            break
        cuts.add(cut)
        k += 1
    cuts = sorted(cuts)
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:])]


def layout_boxes(T, H, W, nt, nh, nw, layout, half="floor"):
    """Window boxes ((t0,t1),(h0,h1),(w0,w1)) in enumeration order.

    CANONICAL is one box covering the grid, so its token order is row-major
    (t, h, w) = canonical id order.
    """
    if layout == CANONICAL:
        return [((0, T), (0, H), (0, W))]
    wt, wh, ww = window_size(T, H, W, nt, nh, nw)
    if layout == REGULAR:
        axis = regular_intervals
    else:
        axis = lambda n, w: shifted_intervals(n, w, half)
    ti, hi, wi = axis(T, wt), axis(H, wh), axis(W, ww)
    boxes = []
    for iw in wi:            # w outermost
        for ih in hi:
            for it in ti:    # t innermost
                boxes.append((it, ih, iw))
    return boxes


def layout_tables(T, H, W, nt, nh, nw, layout, half="floor"):
    """(win_off, ids): window offsets and layout-position -> canonical id.

    ids is obtained by windowing arange(T*H*W).reshape(T, H, W) box by box.
    """
    cube = np.arange(T * H * W, dtype=np.int64).reshape(T, H, W)
    pieces, off = [], [0]
    for (t0, t1), (h0, h1), (w0, w1) in layout_boxes(T, H, W, nt, nh, nw, layout, half):
        piece = cube[t0:t1, h0:h1, w0:w1].reshape(-1)
        pieces.append(piece)
        off.append(off[-1] + piece.size)
    return np.asarray(off, dtype=np.int64), np.concatenate(pieces)


def layer_layout(layer):
    """Layout of a layer in the alternating schedule: regular on even layers."""
    return REGULAR if layer % 2 == 0 else SHIFTED
