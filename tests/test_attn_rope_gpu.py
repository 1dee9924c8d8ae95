"""wp_window_attn_rope (window attention with the window-local RoPE applied
within the call: k rotated once into the workspace, the video Q tiles inside
the attention kernel) against the oracle's RoPE followed by the oracle's
window attention (gpu).

Tolerance: bf16, max abs error <= 2e-2 against the float64 oracle fed the same
un-rotated input bits (Q is rotated in bf16 arithmetic)."""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import plan as op
from oracle import rope as orp

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _oracle(grid, layout, raw, L, base=10000.0, half="floor"):
    pv, pt = orp.positions(*grid, layout, L, half=half)
    q, k = orp.rope(raw["q"], pv, base), orp.rope(raw["k"], pv, base)
    qt, kt = (orp.rope(raw["qt"], pt, base), orp.rope(raw["kt"], pt, base)) if L else (raw["qt"], raw["kt"])
    off, ids = op.layout_tables(*grid, layout, half=half)
    ref_o, ref_t = oa.window_attention(q, k, raw["v"], qt, kt, raw["vt"], off, ids)
    return ref_o, (oa.text_mean(ref_t) if L else None)


@pytest.mark.parametrize("grid,heads,L", [
    ((3, 30, 40, 2, 3, 3), 2, 16),      # ragged windows in both layouts, one text tile
    ((2, 45, 80, 1, 3, 3), 1, 300),     # 720p-like frame, three text tiles (ragged)
    ((5, 16, 24, 2, 1, 1), 3, 0),       # no text; odd window counts
])
def test_rope_attention_matches_oracle(vds, grid, heads, L):
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(N, max(L, 1), heads, 128, torch.bfloat16, "cuda", base_seed=7 * layout)
        raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
        if not L:
            for n in ("qt", "kt", "vt"):
                raw[n] = raw[n][:0]
        before = {n: x[n].clone() for n in ("q", "k", "qt", "kt")}
        o = torch.full((N, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        t = torch.full((max(L, 1), heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
        args = (x["qt"][:L], x["kt"][:L], x["vt"][:L]) if L else (None, None, None)
        vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], *args, o, t[:L] if L else None, ws)
        assert vds.read_status(ws) == 0
        ref_o, ref_t = _oracle(grid, layout, raw, L)
        assert np.abs(_np(o) - ref_o).max() <= TOL, layout
        if L:
            assert np.abs(_np(t[:L]) - ref_t).max() <= TOL, layout
        for n, b in before.items():          # the inputs are not rotated in place
            assert torch.equal(x[n], b), n
    plan.close()


def test_rope_attention_half_ceil_plan(vds):
    """A plan with the other reading of an odd half window (window 2 x 15 x
    27; WP_PLAN_HALF_CEIL): the window-local positions follow the plan's
    boxes, against the oracle's half="ceil" windows and positions."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (2, 45, 80, 1, 3, 3), 2, 16
    plan = vds.Plan(*grid, device="cuda", half="ceil")
    N = plan.N
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(N, L, heads, 128, torch.bfloat16, "cuda", base_seed=9 + layout)
        raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
        o = torch.full((N, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        t = torch.full((L, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
        vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        assert vds.read_status(ws) == 0
        ref_o, ref_t = _oracle(grid, layout, raw, L, half="ceil")
        assert np.abs(_np(o) - ref_o).max() <= TOL, layout
        assert np.abs(_np(t) - ref_t).max() <= TOL, layout
    plan.close()


def test_rope_attention_agrees_with_rope_pass(vds):
    """Same layer through wp_rope + wp_window_attn_to: the two agree within
    the bf16 tolerance, in every output layout."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 40
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    for layout in (op.REGULAR, op.SHIFTED):
        for out_layout in (op.CANONICAL, op.REGULAR, op.SHIFTED):
            x = synth.attention_inputs(N, L, heads, 128, torch.bfloat16, "cuda", base_seed=3)
            o1 = torch.empty((N, heads, 128), dtype=torch.bfloat16, device="cuda")
            t1 = torch.empty((L, heads, 128), dtype=torch.bfloat16, device="cuda")
            ws1 = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
            vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o1, t1, ws1,
                                 out_layout=out_layout)
            assert vds.read_status(ws1) == 0
            vds.rope(plan, layout, x["q"], x["k"], x["qt"], x["kt"])
            o2 = torch.empty_like(o1)
            t2 = torch.empty_like(t1)
            ws2 = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda")
            vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o2, t2, ws2,
                            out_layout=out_layout)
            assert (o1.float() - o2.float()).abs().max().item() <= TOL
            assert (t1.float() - t2.float()).abs().max().item() <= TOL
    plan.close()


@pytest.mark.parametrize("layout", [op.REGULAR, op.SHIFTED])
def test_rope_attention_rotated_k_equals_rope_pass(vds, layout):
    """The call rotates k once into its workspace (documented layout: after
    the status block, the T_w partials and the rotated text q/k, from the
    next multiple of 1024 bytes, [N, heads, 128] bf16).  Both that pass and
    wp_rope rotate in fp32 and round once, so the copy equals wp_rope's k bit
    for bit, and the text q/k copies equal wp_rope's text rows; k itself is
    left as it was.  q/k come packed with v, as a
    projection writes them (row stride 3 * heads * 256 bytes)."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 3, 200
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    g = torch.Generator(device="cuda").manual_seed(11 + layout)
    qkv = torch.randn((N, 3, heads, 128), device="cuda", generator=g).to(torch.bfloat16)
    x = synth.attention_inputs(N, L, heads, 128, torch.bfloat16, "cuda", base_seed=5)
    k_before = qkv[:, 1].clone()
    o = torch.empty((N, heads, 128), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, heads, 128), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
    vds.window_attn_rope(plan, layout, qkv[:, 0], qkv[:, 1], qkv[:, 2], x["qt"], x["kt"], x["vt"], o, t, ws)
    assert vds.read_status(ws) == 0
    assert torch.equal(qkv[:, 1], k_before)
    plain = vds.wp.workspace_bytes(plan, layout, heads, 128, L, vds.BF16)
    off = (plain + 2 * L * heads * 128 * 2 + 1023) // 1024 * 1024
    assert ws.numel() == off + N * heads * 128 * 2
    krot = ws[off:].view(torch.bfloat16).view(N, heads, 128)
    ref = qkv.clone()
    qt_ref, kt_ref = x["qt"].clone(), x["kt"].clone()
    vds.rope(plan, layout, ref[:, 0], ref[:, 1], qt_ref, kt_ref)
    torch.cuda.synchronize()
    assert torch.equal(krot, ref[:, 1])
    # the rotated text q and k, right after the T_w partials, equal wp_rope's too
    tq = ws[plain:plain + L * heads * 256].view(torch.bfloat16).view(L, heads, 128)
    tk = ws[plain + L * heads * 256:plain + 2 * L * heads * 256].view(torch.bfloat16).view(L, heads, 128)
    assert torch.equal(tq, qt_ref) and torch.equal(tk, kt_ref)
    plan.close()


def test_rope_attention_text_stride_and_rejections(vds):
    """Text q/k/v inside a wider buffer (row stride > heads*128*2); then the
    cases the call refuses before launching anything."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 20
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    layout = op.SHIFTED
    x = synth.attention_inputs(N, L, heads, 128, torch.bfloat16, "cuda", base_seed=21)
    wide = torch.zeros((L, 3, heads + 1, 128), dtype=torch.bfloat16, device="cuda")
    wide[:, 0, :heads], wide[:, 1, :heads], wide[:, 2, :heads] = x["qt"], x["kt"], x["vt"]
    qt, kt, vt = wide[:, 0, :heads], wide[:, 1, :heads], wide[:, 2, :heads]
    raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
    o = torch.empty((N, heads, 128), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, heads, 128), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
    vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], qt, kt, vt, o, t, ws)
    assert vds.read_status(ws) == 0
    ref_o, ref_t = _oracle(grid, layout, raw, L)
    assert np.abs(_np(o) - ref_o).max() <= TOL
    assert np.abs(_np(t) - ref_t).max() <= TOL

    small = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda")   # no room for rotated text
    with pytest.raises(vds.wp.WpError) as e:
        vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, small)
    assert e.value.code == 1                                                    # WP_EINVAL
    with pytest.raises(vds.wp.WpError) as e:
        vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws,
                             rope_base=1.0)
    assert e.value.code == 1
    x64 = synth.attention_inputs(N, L, heads, 64, torch.bfloat16, "cuda")
    o64 = torch.empty((N, heads, 64), dtype=torch.bfloat16, device="cuda")
    t64 = torch.empty((L, heads, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vds.wp.WpError) as e:
        vds.window_attn_rope(plan, layout, x64["q"], x64["k"], x64["v"], x64["qt"], x64["kt"], x64["vt"],
                             o64, t64, ws)
    assert e.value.code == 2                                                    # WP_EUNSUPPORTED
    xf = synth.attention_inputs(N, L, heads, 128, torch.float32, "cuda")
    of = torch.empty((N, heads, 128), dtype=torch.float32, device="cuda")
    tf = torch.empty((L, heads, 128), dtype=torch.float32, device="cuda")
    wsf = vds.make_workspace(plan, layout, heads, 128, L, vds.FP32, "cuda", rope=True)
    with pytest.raises(vds.wp.WpError) as e:
        vds.window_attn_rope(plan, layout, xf["q"], xf["k"], xf["v"], xf["qt"], xf["kt"], xf["vt"], of, tf, wsf)
    assert e.value.code == 2
    plan.close()


def test_rope_attention_1080p_sampled(vds):
    """The 1080p-like layer at full size in both layouts, launched as the
    bench launches it: a few (window, head) pairs (first, last, smallest,
    largest and random windows) against the oracle's RoPE followed by its
    window attention, and that head's text output against the oracle's mean
    over every window; every output written and q/k left un-rotated."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L, h = (21, 68, 120, 4, 3, 3), 24, 128, 256, 7
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda")
    before = {n: x[n].clone() for n in ("q", "k", "qt", "kt")}
    rng = np.random.default_rng(2)
    txt = {n: _np(x[n][:, h:h + 1]) for n in ("qt", "kt", "vt")}
    for layout in (op.REGULAR, op.SHIFTED):
        o = torch.full((N, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        t = torch.full((L, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, hd, L, vds.BF16, "cuda", rope=True)
        vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        assert vds.read_status(ws) == 0
        assert not torch.isnan(o).any() and not torch.isnan(t).any()
        off, ids = op.layout_tables(*grid, layout)
        nwin, sizes = len(off) - 1, np.diff(off)
        wins = sorted({0, nwin - 1, int(sizes.argmin()), int(sizes.argmax())} |
                      set(rng.choice(nwin, size=3, replace=False).tolist()))
        rows = np.concatenate([np.arange(off[w], off[w + 1]) for w in wins])
        sel = torch.from_numpy(rows).cuda()
        pv, pt = orp.positions(*grid, layout, L)
        q = orp.rope(_np(x["q"][sel, h:h + 1]), pv[rows])
        k = orp.rope(_np(x["k"][sel, h:h + 1]), pv[rows])
        v = _np(x["v"][sel, h:h + 1])
        qt, kt = orp.rope(txt["qt"], pt), orp.rope(txt["kt"], pt)
        sub_off = np.concatenate([[0], np.cumsum(sizes[wins])])
        ref_o, ref_t = oa.window_attention(q, k, v, qt, kt, txt["vt"], sub_off, np.arange(rows.size))
        got = _np(o[torch.from_numpy(ids[rows]).cuda(), h:h + 1])
        assert np.abs(got - ref_o).max() <= TOL, layout
        # the text output of head h: every window's rotated text queries
        # against [its rotated video keys ; rotated text keys], averaged
        kh = orp.rope(_np(x["k"][:, h:h + 1]), pv)[:, 0]
        vh = _np(x["v"][:, h:h + 1])[:, 0]
        t_win = np.empty((nwin, L, 1, hd))
        for w in range(nwin):
            a, b = int(off[w]), int(off[w + 1])
            t_win[w, :, 0] = oa.segment_attention(qt[:, 0], np.concatenate([kh[a:b], kt[:, 0]]),
                                                  np.concatenate([vh[a:b], txt["vt"][:, 0]]), 1.0 / np.sqrt(hd))
        assert np.abs(_np(t[:, h]) - oa.text_mean(t_win)[:, 0]).max() <= TOL, layout
    for n, b in before.items():
        assert torch.equal(x[n], b), n
    plan.close()


def _random_cases(n, seed=37):
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        grid = (rng.randint(1, 4), rng.randint(4, 40), rng.randint(4, 60),
                rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 4))
        if min(op.window_size(*grid)) < 1 or sum(op.window_size(*grid)) > 196:
            continue
        out.append((grid, rng.randint(1, 3), rng.choice([0, 1, 7, 130]), rng.choice([op.REGULAR, op.SHIFTED]),
                    rng.choice([op.CANONICAL, op.REGULAR, op.SHIFTED])))
    return out


@pytest.mark.parametrize("grid,heads,L,layout,out", _random_cases(5))
def test_rope_attention_random_configs(vds, grid, heads, L, layout, out):
    """Seeded random grids, window counts, head counts, text lengths, layouts
    and output layouts, against the oracle's RoPE followed by its attention."""
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, max(L, 1), heads, 128, torch.bfloat16, "cuda", base_seed=sum(grid))
    raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
    if not L:
        for n in ("qt", "kt", "vt"):
            raw[n] = raw[n][:0]
    o = torch.full((N, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    t = torch.full((max(L, 1), heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda", rope=True)
    args = (x["qt"][:L], x["kt"][:L], x["vt"][:L]) if L else (None, None, None)
    vds.window_attn_rope(plan, layout, x["q"], x["k"], x["v"], *args, o, t[:L] if L else None, ws, out_layout=out)
    assert vds.read_status(ws) == 0
    ref_o, ref_t = _oracle(grid, layout, raw, L)
    got = _np(o)
    if out != op.CANONICAL:
        got = got[np.argsort(op.layout_tables(*grid, out)[1])]
    assert np.abs(got - ref_o).max() <= TOL
    if L:
        assert np.abs(_np(t[:L]) - ref_t).max() <= TOL
    plan.close()
