"""Pins for the oracle's window attention and text mean (CPU only).

The oracle is checked against a library routine (torch's scaled-dot-product
attention in float64, a different implementation of the same textbook
formula), against closed forms (q = 0 gives the segment mean of V; the text
mean of §Text stream then has a closed form that separates a per-window mean
from a token-weighted one), against the page's "one window covering the grid
is global attention" special case, and against invariants (a permutation of
the keys inside a window changes nothing; a dominant key selects its value).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as oa
from oracle import plan as op


def _inputs(N, L, heads, hd, seed):
    rng = np.random.default_rng(seed)
    mk = lambda n: rng.standard_normal((n, heads, hd))
    return mk(N), mk(N), mk(N), mk(L), mk(L), mk(L)


def _sdpa(Q, K, V, scale=None):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))[None, None]
    return F.scaled_dot_product_attention(t(Q), t(K), t(V), scale=scale)[0, 0].numpy()


@pytest.mark.parametrize("layout", [op.REGULAR, op.SHIFTED])
@pytest.mark.parametrize("grid,heads,hd,L", [((3, 30, 40, 2, 3, 3), 2, 16, 5),
                                             ((3, 7, 11, 2, 2, 3), 3, 8, 0),
                                             ((2, 45, 80, 1, 3, 3), 1, 8, 16)])
def test_matches_torch_sdpa_per_window(layout, grid, heads, hd, L):
    off, ids = op.layout_tables(*grid, layout)
    N = ids.size
    q, k, v, qt, kt, vt = _inputs(N, L, heads, hd, seed=1)
    o_vid, t_win = oa.window_attention(q, k, v, qt, kt, vt, off, ids)
    assert not np.isnan(o_vid).any()
    for w in range(len(off) - 1):
        a, b = off[w], off[w + 1]
        for h in range(heads):
            Q = np.concatenate([q[a:b, h], qt[:, h]])
            K = np.concatenate([k[a:b, h], kt[:, h]])
            V = np.concatenate([v[a:b, h], vt[:, h]])
            Y = _sdpa(Q, K, V)
            # video rows land at their canonical ids: token ids[a+i]
            np.testing.assert_allclose(o_vid[ids[a:b], h], Y[: b - a], rtol=0, atol=1e-12)
            np.testing.assert_allclose(t_win[w, :, h], Y[b - a:], rtol=0, atol=1e-12)


def test_single_window_is_global_attention():
    """One window covering the grid (nt=nh=nw=1, H*W <= 3600, T <= 30):
    both layouts are plain global attention over [all video ; text]."""
    T, H, W = 3, 9, 16
    assert op.window_size(T, H, W, 1, 1, 1) == (3, 45, 80)  # covers 9x16
    heads, hd, L = 2, 16, 7
    rng = np.random.default_rng(3)
    Xc = [rng.standard_normal((T * H * W, heads, hd)) for _ in range(3)]
    Xt = [rng.standard_normal((L, heads, hd)) for _ in range(3)]
    for layout in (op.REGULAR, op.SHIFTED):
        off, ids = op.layout_tables(T, H, W, 1, 1, 1, layout)
        assert len(off) == 2
        # inputs are in layout order: row p holds canonical token ids[p]
        q, k, v = (x[ids] for x in Xc)
        o_vid, t_win = oa.window_attention(q, k, v, *Xt, off, ids)
        for h in range(heads):
            Y = _sdpa(*(np.concatenate([Xc[i][:, h], Xt[i][:, h]]) for i in range(3)))
            np.testing.assert_allclose(o_vid[:, h], Y[: T * H * W], atol=1e-12, rtol=0)
            np.testing.assert_allclose(oa.text_mean(t_win)[:, h], Y[T * H * W:],
                                       atol=1e-12, rtol=0)


def test_zero_queries_give_segment_mean_and_text_mean_closed_form():
    """q = 0 makes every score 0, so each output row is the plain mean of V
    over its segment [window ; text].  Then §Text stream's
    T_next = (sum_w T_w) / nwin has the closed form below; the windows are
    ragged, so a token-weighted mean or a mean of a different count would
    differ from it."""
    grid = (2, 45, 80, 1, 3, 3)
    heads, hd, L = 2, 4, 16
    for layout in (op.REGULAR, op.SHIFTED):
        off, ids = op.layout_tables(*grid, layout)
        N = ids.size
        _, k, v, _, kt, vt = _inputs(N, L, heads, hd, seed=5)
        q = np.zeros((N, heads, hd))
        qt = np.zeros((L, heads, hd))
        o_vid, t_win = oa.window_attention(q, k, v, qt, kt, vt, off, ids)
        nwin = len(off) - 1
        seg_means = []
        for w in range(nwin):
            a, b = off[w], off[w + 1]
            m = (v[a:b].sum(axis=0) + vt.sum(axis=0)) / (b - a + L)   # [heads, hd]
            seg_means.append(m)
            np.testing.assert_allclose(o_vid[ids[a:b]], np.broadcast_to(m, (b - a, heads, hd)),
                                       atol=1e-12, rtol=0)
        expect = sum(seg_means) / nwin
        got = oa.text_mean(t_win)
        np.testing.assert_allclose(got, np.broadcast_to(expect, (L, heads, hd)), atol=1e-12, rtol=0)
        sizes = np.diff(off) + L
        token_weighted = sum(m * s for m, s in zip(seg_means, sizes)) / sizes.sum()
        assert np.abs(got[0] - token_weighted).max() > 1e-6


def test_key_permutation_inside_window_is_invariant():
    grid = (3, 30, 40, 2, 3, 3)
    off, ids = op.layout_tables(*grid, op.SHIFTED)
    q, k, v, qt, kt, vt = _inputs(ids.size, 3, 2, 8, seed=9)
    o1, t1 = oa.window_attention(q, k, v, qt, kt, vt, off, ids)
    # reorder rows inside window 0 (keys and values together, and the id table)
    a, b = off[0], off[1]
    perm = np.arange(ids.size)
    perm[a:b] = a + np.random.default_rng(0).permutation(b - a)
    o2, t2 = oa.window_attention(q[perm], k[perm], v[perm], qt, kt, vt, off, ids[perm])
    np.testing.assert_allclose(o1, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(t1, t2, atol=1e-12, rtol=0)


def test_dominant_key_selects_its_value():
    """Scores of one key far above the rest: the softmax puts all its weight
    there, so the output is that key's value row (video or text key)."""
    grid = (1, 4, 4, 1, 1, 1)      # window covers the grid
    off, ids = op.layout_tables(*grid, op.REGULAR)
    N, heads, hd, L = ids.size, 1, 8, 2
    q, k, v, qt, kt, vt = _inputs(N, L, heads, hd, seed=2)
    e = np.zeros(hd); e[3] = 1.0
    q[:] = 50.0 * e; qt[:] = 50.0 * e
    k[:, :, 3] = 0.0; kt[:, :, 3] = 0.0
    k[5, 0, 3] = 10.0                # video key row 5 (layout order) dominates
    o, t = oa.window_attention(q, k, v, qt, kt, vt, off, ids, scale=1.0)
    np.testing.assert_allclose(o[:, 0], np.broadcast_to(v[5, 0], (N, hd)), atol=1e-12)
    np.testing.assert_allclose(t[0, :, 0], np.broadcast_to(v[5, 0], (L, hd)), atol=1e-12)
    k[5, 0, 3] = 0.0
    kt[1, 0, 3] = 10.0               # now text key 1 dominates
    o, t = oa.window_attention(q, k, v, qt, kt, vt, off, ids, scale=1.0)
    np.testing.assert_allclose(o[:, 0], np.broadcast_to(vt[1, 0], (N, hd)), atol=1e-12)


def test_scale_argument_and_default():
    grid = (1, 3, 5, 1, 1, 1)
    off, ids = op.layout_tables(*grid, op.REGULAR)
    q, k, v, qt, kt, vt = _inputs(ids.size, 4, 1, 16, seed=4)
    o_def, _ = oa.window_attention(q, k, v, qt, kt, vt, off, ids)
    o_exp, _ = oa.window_attention(q, k, v, qt, kt, vt, off, ids, scale=1 / math.sqrt(16))
    np.testing.assert_array_equal(o_def, o_exp)
    o_s, _ = oa.window_attention(q, k, v, qt, kt, vt, off, ids, scale=0.3)
    Y = _sdpa(*(np.concatenate([x[:, 0], y[:, 0]]) for x, y in ((q[ids.argsort()], qt), (k[ids.argsort()], kt), (v[ids.argsort()], vt))), scale=0.3)
    np.testing.assert_allclose(o_s[:, 0], Y[: ids.size], atol=1e-12, rtol=0)


def test_subset_leaves_other_entries_nan():
    grid = (3, 30, 40, 2, 3, 3)
    off, ids = op.layout_tables(*grid, op.REGULAR)
    q, k, v, qt, kt, vt = _inputs(ids.size, 3, 3, 8, seed=6)
    full_o, full_t = oa.window_attention(q, k, v, qt, kt, vt, off, ids)
    o, t = oa.window_attention(q, k, v, qt, kt, vt, off, ids, windows=[1], heads=[2])
    a, b = off[1], off[2]
    np.testing.assert_array_equal(o[ids[a:b], 2], full_o[ids[a:b], 2])
    np.testing.assert_array_equal(t[1, :, 2], full_t[1, :, 2])
    assert np.isnan(o[ids[a:b], 0]).all() and np.isnan(t[0]).all()
