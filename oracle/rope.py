"""Oracle window-local 3D rotary position embedding (test infrastructure;
see the package docstring).

"Window-Aligned Sequence Parallelism (SeedVR2)", §Reference quirks
reproduced on purpose: RoPE positions are window-local -- a video token at
window-local (dt, dh, dw) uses axial indices (text_len + dt, dh, dw), and
every window restarts at 0; the rotary span is 3 * (rope_dim // 3) channels
(126 of 128), so the last two channels pass through unrotated.

Readings of what the page leaves open:
* the span is three equal blocks, axes t, h, w in that order (42 channels
  each at head_dim 128);
* inside a block of d channels, channels (2i, 2i+1) form a pair rotated by
  the angle pos * base**(-2i/d), base 10000 (the usual RoPE frequencies);
* a text token at position l uses the axial indices (l, l, l) -- one
  position on every axis, the usual way a 1-D sequence enters a multi-axis
  rotary scheme; the page's offset of the video t axis by text_len then
  places every video token after the text.
Computed in float64.
"""
import numpy as np

from . import plan as op


def positions(T, H, W, nt, nh, nw, layout, L, half="floor"):
    """(pos_video [N, 3] in layout row order, pos_text [L, 3]); half as in
    plan.layout_boxes."""
    rows = []
    for (t0, t1), (h0, h1), (w0, w1) in op.layout_boxes(T, H, W, nt, nh, nw, layout, half):
        for t in range(t0, t1):          # row-major (t, h, w) inside a window
            for h in range(h0, h1):
                for w in range(w0, w1):
                    rows.append((L + (t - t0), h - h0, w - w0))
    pos_txt = np.array([(l, l, l) for l in range(L)], dtype=np.float64).reshape(L, 3)
    return np.array(rows, dtype=np.float64).reshape(-1, 3), pos_txt


def rope(x, pos, base=10000.0):
    """Rotate x [n, heads, head_dim] by the axial positions pos [n, 3]."""
    x = np.array(x, dtype=np.float64)
    hd = x.shape[-1]
    d = hd // 3                      # channels per axis; the span is 3*d
    out = x.copy()
    for a in range(3):
        for i in range(d // 2):
            c0 = a * d + 2 * i
            ang = pos[:, a] * base ** (-2.0 * i / d)          # [n]
            cos, sin = np.cos(ang)[:, None], np.sin(ang)[:, None]
            x0, x1 = x[:, :, c0], x[:, :, c0 + 1]
            out[:, :, c0] = x0 * cos - x1 * sin
            out[:, :, c0 + 1] = x0 * sin + x1 * cos
    return out
