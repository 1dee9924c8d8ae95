"""Oracle window attention and text mean (test infrastructure).

"Window-Aligned Sequence Parallelism (SeedVR2)":

* §SeedVR2 integration -- each layer runs one attention per segment
  ``[video tokens of one window ; the replicated text tokens]``; the segments
  are independent and attention inside a segment is full (bidirectional, no
  mask).  The video outputs go back to canonical token order.
* §Text stream -- every window produces its own text output ``T_w``; the
  next text state is ``(sum over windows of T_w) / (number of windows of the
  current layout)`` -- a plain sum over windows, not a token-weighted mean.

Arithmetic: inputs are converted to float64 and every product, exponential
and sum is taken in float64, in the order written.  The softmax scale is
``1/sqrt(head_dim)`` unless given (the page does not state it; this is the
usual scaled-dot-product default).

Video inputs q, k, v are ``[N, heads, head_dim]`` in the layout's row order
(rows ``win_off[w] .. win_off[w+1]`` are window w); text inputs are
``[L, heads, head_dim]``.  ``ids`` maps layout row -> canonical token id.
"""
import math

import numpy as np


def segment_attention(Q, K, V, scale):
    """softmax(Q K^T * scale) V for one segment and one head, in float64."""
    S = (Q @ K.T) * scale
    S = S - S.max(axis=1, keepdims=True)
    P = np.exp(S)
    P = P / P.sum(axis=1, keepdims=True)
    return P @ V


def window_attention(q, k, v, qt, kt, vt, win_off, ids, scale=None,
                     windows=None, heads=None):
    """Per-window attention over [video window ; text].

    Returns ``(o_vid, t_win)``: ``o_vid[N, heads, hd]`` in canonical order and
    ``t_win[nwin, L, heads, hd]``, the text output of every window.  With
    ``windows``/``heads`` given, only those (window, head) pairs are computed
    and every other entry is NaN.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    qt, kt, vt = (np.asarray(x, dtype=np.float64) for x in (qt, kt, vt))
    N, nheads, hd = q.shape
    L = qt.shape[0]
    nwin = len(win_off) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    o_vid = np.full((N, nheads, hd), np.nan)
    t_win = np.full((nwin, L, nheads, hd), np.nan)
    for w in (range(nwin) if windows is None else windows):
        a, b = int(win_off[w]), int(win_off[w + 1])
        for h in (range(nheads) if heads is None else heads):
            Q = np.concatenate([q[a:b, h], qt[:, h]])
            K = np.concatenate([k[a:b, h], kt[:, h]])
            V = np.concatenate([v[a:b, h], vt[:, h]])
            Y = segment_attention(Q, K, V, scale)
            o_vid[ids[a:b], h] = Y[: b - a]
            t_win[w, :, h] = Y[b - a:]
    return o_vid, t_win


def text_mean(t_win):
    """(T_0 + T_1 + ... + T_{nwin-1}) / nwin, summed in enumeration order."""
    acc = np.zeros(t_win.shape[1:], dtype=np.float64)
    for w in range(t_win.shape[0]):
        acc = acc + t_win[w]
    return acc / t_win.shape[0]
