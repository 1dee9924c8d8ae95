"""wp_window_attn on the GPU against the oracle (gpu).

Tolerances: max abs error <= 1e-4 in fp32 mode and <= 2e-2 in bf16 mode,
against the float64 oracle fed the same input bits.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import plan as op

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _run(vds, plan, layout, x, heads, hd, L, dtype, scale=0.0):
    N = plan.N
    dev = x["q"].device
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    o_vid = torch.full((N, heads, hd), float("nan"), dtype=dtype, device=dev)
    o_txt = torch.full((L, heads, hd), float("nan"), dtype=dtype, device=dev)
    ws = vds.make_workspace(plan, layout, heads, hd, L, code, dev)
    vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o_vid, o_txt, ws,
                    scale=scale)
    assert vds.read_status(ws) == 0
    return o_vid, o_txt, ws


def _check_full(vds, grid, heads, hd, L, dtype, layouts=(op.REGULAR, op.SHIFTED), scale=0.0, half="floor"):
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda", half=half)
    N = plan.N
    for layout in layouts:
        x = synth.attention_inputs(N, L, heads, hd, dtype, "cuda", base_seed=10 * layout)
        o_vid, o_txt, _ = _run(vds, plan, layout, x, heads, hd, L, dtype, scale)
        off, ids = op.layout_tables(*grid, layout, half=half)
        ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids,
                                           scale=scale if scale > 0 else None)
        err_v = np.abs(_np(o_vid) - ref_o).max()
        assert err_v <= TOL[dtype], (layout, err_v)
        if L:
            err_t = np.abs(_np(o_txt) - oa.text_mean(ref_t)).max()
            assert err_t <= TOL[dtype], (layout, err_t)
    plan.close()


def test_pr1_fp32(vds):
    """T=2, H=45, W=80, nt=1, nh=nw=3; heads 2, head_dim 64, L 16, fp32."""
    _check_full(vds, (2, 45, 80, 1, 3, 3), 2, 64, 16, torch.float32)


@pytest.mark.parametrize("hd", [64, 128])
def test_pr1_grid_bf16(vds, hd):
    _check_full(vds, (2, 45, 80, 1, 3, 3), 2, hd, 16, torch.bfloat16)


@pytest.mark.parametrize("L", [0, 1, 128, 300])
def test_text_lengths_bf16(vds, L):
    """No text, one token, exactly one tile, and a ragged third tile."""
    _check_full(vds, (3, 30, 40, 2, 3, 3), 2, 128, L, torch.bfloat16)


@pytest.mark.parametrize("L", [0, 5, 300])
def test_text_lengths_fp32(vds, L):
    _check_full(vds, (3, 30, 40, 2, 3, 3), 3, 128, L, torch.float32)


def test_single_window_is_global_attention(vds):
    """One window covers the grid: global attention over [video ; text]."""
    _check_full(vds, (3, 9, 16, 1, 1, 1), 2, 128, 7, torch.bfloat16)
    _check_full(vds, (3, 9, 16, 1, 1, 1), 2, 64, 7, torch.float32)


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_half_ceil_plan(vds, dtype, hd):
    """A plan made with the other reading of an odd half window
    (WP_PLAN_HALF_CEIL) against the oracle's half="ceil" windows: attention
    in both layouts, and the re-layout between them bit for bit."""
    from oracle import permute as opm
    grid = (2, 45, 80, 1, 3, 3)           # window 2 x 15 x 27: odd on both spatial axes
    _check_full(vds, grid, 2, hd, 40, dtype, half="ceil")
    plan = vds.Plan(*grid, device="cuda", half="ceil")
    rows = torch.randint(-2 ** 15, 2 ** 15, (plan.N, 48), dtype=torch.int16, device="cuda")
    out = torch.empty_like(rows)
    vds.permute(plan, rows, out, vds.REGULAR, vds.SHIFTED)
    torch.cuda.synchronize()
    ids = {l: op.layout_tables(*grid, l, half="ceil")[1] for l in (op.REGULAR, op.SHIFTED)}
    assert np.array_equal(out.cpu().numpy(), opm.permute_rows(rows.cpu().numpy(), ids[op.REGULAR], ids[op.SHIFTED]))
    plan.close()


def test_custom_scale(vds):
    _check_full(vds, (2, 45, 80, 1, 3, 3), 1, 128, 16, torch.bfloat16, layouts=(op.SHIFTED,), scale=0.05)


def test_tiny_windows_and_tail_past_n(vds):
    """Windows of a few tokens (tiles mostly padding); the last window's tile
    runs past row N (zero-filled by TMA)."""
    _check_full(vds, (2, 45, 80, 1, 9, 16), 2, 128, 3, torch.bfloat16)   # 50-token windows, 8 shifted
    _check_full(vds, (2, 3, 200, 1, 1, 9), 1, 64, 0, torch.bfloat16)


def _windows_to_check(off, boxes, rng, small=1300):
    """First, last and largest window, one window of every distinct box
    shape up to `small` tokens (the clipped edge classes of the shifted
    layout: 1-row h-slices, the 39-token corner, ...), and one random window."""
    nwin, sizes = len(off) - 1, np.diff(off)
    wins = {0, nwin - 1, int(sizes.argmax()), int(rng.integers(nwin))}
    seen = set()
    for w, b in enumerate(boxes):
        shape = tuple(x1 - x0 for x0, x1 in b)
        if shape not in seen and sizes[w] <= small:
            seen.add(shape)
            wins.add(w)
    return sorted(wins)


def _oracle_text_mean(x, off, heads):
    """The oracle's text output for the given heads: every window's text
    query rows attend to [that window's video rows ; text] (§Text stream),
    and the per-window results are averaged over all windows in order."""
    L, hd = x["qt"].shape[0], x["qt"].shape[2]
    out = {}
    for h in heads:
        k, v = _np(x["k"][:, h]), _np(x["v"][:, h])
        qt, kt, vt = (_np(x[n][:, h]) for n in ("qt", "kt", "vt"))
        t_win = np.empty((len(off) - 1, L, 1, hd))
        for w in range(len(off) - 1):
            a, b = int(off[w]), int(off[w + 1])
            t_win[w, :, 0] = oa.segment_attention(qt, np.concatenate([k[a:b], kt]), np.concatenate([v[a:b], vt]),
                                                  1.0 / np.sqrt(hd))
        out[h] = oa.text_mean(t_win)[:, 0]
    return out


def _sampled_check(vds, grid, heads, hd, L, text_heads=(0,)):
    """Full-size run, launched as the bench launches it.  The oracle computes
    every head of the windows _windows_to_check picks, and the text output
    of `text_heads` over all windows; every video row of the output must be
    written (no NaN left)."""
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda")
    rng = np.random.default_rng(1)
    txt = [_np(x[n]) for n in ("qt", "kt", "vt")]
    for layout in (op.REGULAR, op.SHIFTED):
        o_vid, o_txt, ws = _run(vds, plan, layout, x, heads, hd, L, torch.bfloat16)
        assert not torch.isnan(o_vid).any() and not torch.isnan(o_txt).any()
        off, ids = op.layout_tables(*grid, layout)
        sizes = np.diff(off)
        wins = _windows_to_check(off, op.layout_boxes(*grid, layout), rng)
        rows = np.concatenate([np.arange(off[w], off[w + 1]) for w in wins])
        sel = torch.from_numpy(rows).cuda()
        sub_off = np.concatenate([[0], np.cumsum(sizes[wins])])
        ref_o, _ = oa.window_attention(_np(x["q"][sel]), _np(x["k"][sel]), _np(x["v"][sel]), *txt, sub_off,
                                       np.arange(rows.size))
        got = _np(o_vid[torch.from_numpy(ids[rows]).cuda()])
        err = np.abs(got - ref_o).max(axis=(1, 2))
        for i, w in enumerate(wins):
            e = err[sub_off[i]:sub_off[i + 1]].max()
            assert e <= 2e-2, (layout, w, sizes[w], e)
        ref_t = _oracle_text_mean(x, off, text_heads)
        for h in text_heads:
            assert np.abs(_np(o_txt[:, h]) - ref_t[h]).max() <= 2e-2, (layout, h)
    plan.close()


def test_720p_sampled(vds):
    _sampled_check(vds, (21, 45, 80, 4, 3, 3), 24, 128, 256, text_heads=(0, 23))


def test_1080p_sampled(vds):
    _sampled_check(vds, (21, 68, 120, 4, 3, 3), 24, 128, 256, text_heads=(5, 17))


def test_full_schedule_grid_sampled(vds):
    """The 32-layer schedule's grid (T=30, 90x160: 432,000 tokens, windows of
    8x15x27, 144 regular and 245 shifted) at full size."""
    _sampled_check(vds, (30, 90, 160, 4, 3, 3), 24, 128, 256, text_heads=(11,))


@pytest.mark.parametrize("L", [0, 5])
def test_single_token_grid(vds, L):
    """T = H = W = 1: one window holding one token.  Without text its only
    key is itself, so the output is its own v row exactly (p = 1); with text
    it is the oracle's attention over [1 video ; L text] keys."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd = (1, 1, 1, 1, 1, 1), 3, 128
    plan = vds.Plan(*grid, device="cuda")
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(1, max(L, 1), heads, hd, torch.bfloat16, "cuda", base_seed=29)
        qt, kt, vt = (x["qt"], x["kt"], x["vt"]) if L else (None, None, None)
        o = torch.full((1, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        t = torch.full((max(L, 1), heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, hd, L, vds.BF16, "cuda")
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], qt, kt, vt, o, t[:L] if L else None, ws)
        assert vds.read_status(ws) == 0
        if L == 0:
            assert torch.equal(o, x["v"])
        else:
            off, ids = op.layout_tables(*grid, layout)
            ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
            assert np.abs(_np(o) - ref_o).max() <= TOL[torch.bfloat16]
            assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL[torch.bfloat16]
    plan.close()


def test_bad_alignment_rejected(vds):
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    from video_dit_shifted_gb300 import synth
    x = synth.attention_inputs(plan.N, 16, 2, 96, torch.bfloat16, "cuda")
    o = torch.empty((plan.N, 2, 96), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((16, 2, 96), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(vds.wp.WpError) as e:
        vds.window_attn(plan, op.REGULAR, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
    assert e.value.code == 2
    plan.close()


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_output_in_another_layout_is_attention_then_permute(vds, dtype, hd):
    """Writing the video output straight into layout b equals writing it in
    canonical order and re-laying it out canonical -> b, bit for bit."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 20
    plan = vds.Plan(*grid, device="cuda")
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda", base_seed=3 + layout)
        ws = vds.make_workspace(plan, layout, heads, hd, L, code, "cuda")
        t = torch.empty((L, heads, hd), dtype=dtype, device="cuda")
        canon = torch.empty((plan.N, heads, hd), dtype=dtype, device="cuda")
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], canon, t, ws)
        for out in (op.REGULAR, op.SHIFTED, op.CANONICAL):
            o = torch.full_like(canon, float("nan"))
            vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws,
                            out_layout=out)
            want = torch.empty_like(canon)
            vds.permute(plan, canon.view(plan.N, -1), want.view(plan.N, -1), op.CANONICAL, out)
            assert torch.equal(o, want), (layout, out)
    plan.close()


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
def test_output_in_another_layout_matches_oracle(vds, dtype, hd):
    """wp_window_attn_to against the oracle for every (layout, out_layout)
    pair: the oracle's window attention (video rows in canonical order)
    re-laid out canonical -> out_layout by the oracle's permutation
    ("Window-Aligned Sequence Parallelism (SeedVR2)", §Motivation: at SP=1
    the next layer's layout is a local permutation)."""
    from oracle import permute as opm
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 20
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    canon_ids = np.arange(N)
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(N, L, heads, hd, dtype, "cuda", base_seed=9 + layout)
        off, ids = op.layout_tables(*grid, layout)
        ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        ws = vds.make_workspace(plan, layout, heads, hd, L, code, "cuda")
        for out in (op.CANONICAL, op.REGULAR, op.SHIFTED):
            o = torch.full((N, heads, hd), float("nan"), dtype=dtype, device="cuda")
            t = torch.full((L, heads, hd), float("nan"), dtype=dtype, device="cuda")
            vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws,
                            out_layout=out)
            assert vds.read_status(ws) == 0
            want = opm.permute_rows(ref_o, canon_ids, op.layout_tables(*grid, out)[1])
            assert np.abs(_np(o) - want).max() <= TOL[dtype], (layout, out)
            assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL[dtype], (layout, out)
    plan.close()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_more_than_30_frames(vds, dtype):
    """T > 30: the temporal window is capped at ceil(30/nt), so the regular
    layout has more t windows than nt."""
    grid = (33, 6, 8, 2, 1, 1)
    assert op.window_size(*grid)[0] == 15
    _check_full(vds, grid, 2, 128 if dtype == torch.bfloat16 else 64, 9, dtype)


def test_long_odd_text(vds):
    """L = 520: five text tiles, the last one ragged; three heads."""
    _check_full(vds, (2, 20, 30, 1, 2, 2), 3, 128, 520, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_separate_tensors_and_strided_output(vds, dtype):
    """q, k, v as separate contiguous tensors; o_vid rows inside a wider
    buffer (row stride larger than heads * head_dim); guard columns stay
    untouched."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 16
    hd = 128 if dtype == torch.bfloat16 else 64
    plan = vds.Plan(*grid, device="cuda")
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda", base_seed=11, packed=False)
        wide = torch.full((plan.N, heads + 1, hd), 7.0, dtype=dtype, device="cuda")
        o = wide[:, :heads]                     # row stride (heads + 1) * hd
        t = torch.empty((L, heads, hd), dtype=dtype, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, hd, L, code, "cuda")
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        assert vds.read_status(ws) == 0
        off, ids = op.layout_tables(*grid, layout)
        ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        assert np.abs(_np(o) - ref_o).max() <= TOL[dtype]
        assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL[dtype]
        assert torch.all(wide[:, heads] == 7.0)
    plan.close()


def test_layer_pair_replays_in_a_cuda_graph(vds):
    """attention (regular) -> re-layout -> attention (shifted), captured once
    in a CUDA graph and replayed, gives the eager results bit for bit."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (3, 30, 40, 2, 3, 3), 2, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda")
    qkv_shf = torch.empty_like(x["vid_buf"])
    outs = {l: torch.empty((N, heads, hd), dtype=torch.bfloat16, device="cuda") for l in (op.REGULAR, op.SHIFTED)}
    txt = {l: torch.empty((L, heads, hd), dtype=torch.bfloat16, device="cuda") for l in (op.REGULAR, op.SHIFTED)}
    ws = {l: vds.make_workspace(plan, l, heads, hd, L, vds.BF16, "cuda") for l in (op.REGULAR, op.SHIFTED)}

    def layer_pair():
        b = x["vid_buf"]
        vds.window_attn(plan, op.REGULAR, b[:, 0], b[:, 1], b[:, 2], x["qt"], x["kt"], x["vt"],
                        outs[op.REGULAR], txt[op.REGULAR], ws[op.REGULAR])
        vds.permute(plan, b.view(N, -1), qkv_shf.view(N, -1), op.REGULAR, op.SHIFTED)
        vds.window_attn(plan, op.SHIFTED, qkv_shf[:, 0], qkv_shf[:, 1], qkv_shf[:, 2], x["qt"], x["kt"],
                        x["vt"], outs[op.SHIFTED], txt[op.SHIFTED], ws[op.SHIFTED])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer_pair()                                   # eager, on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (outs[op.REGULAR], outs[op.SHIFTED], txt[op.REGULAR], txt[op.SHIFTED])]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer_pair()
    for t in list(outs.values()) + list(txt.values()):
        t.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for got, want in zip((outs[op.REGULAR], outs[op.SHIFTED], txt[op.REGULAR], txt[op.SHIFTED]), eager):
        assert torch.equal(got, want)
    plan.close()


def test_outputs_aligned_to_16_bytes_only(vds):
    """o_vid starting 16 bytes into its buffer with a row stride of 16 mod 32
    bytes, and a workspace 16 bytes past a 32-byte boundary: the epilogue
    takes its 16-byte store path; results and guard bytes as usual."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (3, 30, 40, 2, 3, 3), 2, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    stride = heads * hd + 8                     # elements: 528 bytes per row
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda", base_seed=13)
        buf = torch.full((N * stride + 16,), 7.0, dtype=torch.bfloat16, device="cuda")
        o = buf[8:].as_strided((N, heads, hd), (stride, hd, 1))
        assert o.data_ptr() % 32 == 16 and (stride * 2) % 32 == 16
        t = torch.empty((L, heads, hd), dtype=torch.bfloat16, device="cuda")
        need = vds.workspace_bytes(plan, layout, heads, hd, L, vds.BF16)
        ws_buf = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
        skip = (16 - ws_buf.data_ptr()) % 32
        ws = ws_buf[skip:skip + need]
        assert ws.data_ptr() % 32 == 16
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        assert vds.read_status(ws) == 0
        off, ids = op.layout_tables(*grid, layout)
        ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        assert np.abs(_np(o) - ref_o).max() <= TOL[torch.bfloat16]
        assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL[torch.bfloat16]
        guard = buf[:8].float()
        assert torch.all(guard == 7.0)
        gaps = buf[8:8 + N * stride].view(N, stride)[:, heads * hd:]
        assert torch.all(gaps.float() == 7.0)
    plan.close()


def test_softmax_slow_paths(vds):
    """Scores built so that every branch of the lazy rescale runs: the first
    tile's max lies outside its first 16 columns (row sum > 2^8 at j = 0:
    the true max is taken and the pass redone), a later tile sits ~3.8 log2
    units above the running max (row sum > 2^8, max within 2^8: redone
    without a rescale), and one key is ~25 log2 units higher still (O and l
    rescaled).  One window of 10 video tiles; checked against the oracle."""
    grid, heads, hd, L = (2, 16, 40, 1, 1, 1), 2, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    off, ids = op.layout_tables(*grid, op.REGULAR)
    assert len(off) == 2 and N == 1280                 # one window, keys in layout order
    g = torch.Generator().manual_seed(5)
    b = torch.randn(N, generator=g) * 4.0               # score of key n = b[n] (q = e_0)
    b[:128] = 0.0
    b[20] = 100.0                                       # tile 0: max outside the first 16 columns
    b[128:256] = 130.0                                  # tile 1: every p ~ 2^3.8 over the running max
    b[300] = 300.0                                      # tile 2: ~25 log2 units higher: rescale
    q = torch.zeros(N, heads, hd)
    q[:, :, 0] = 1.0
    k = torch.zeros(N, heads, hd)
    k[:, :, 0] = b[:, None]
    v = torch.randn(N, heads, hd, generator=g)
    qt = torch.randn(L, heads, hd, generator=g) * 0.1
    kt = torch.randn(L, heads, hd, generator=g)
    vt = torch.randn(L, heads, hd, generator=g)
    x = {n: t.to(torch.bfloat16).cuda() for n, t in dict(q=q, k=k, v=v, qt=qt, kt=kt, vt=vt).items()}
    o = torch.full((N, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    t = torch.full((L, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, op.REGULAR, heads, hd, L, vds.BF16, "cuda")
    vds.window_attn(plan, op.REGULAR, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
    assert vds.read_status(ws) == 0
    ref_o, ref_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
    assert np.abs(_np(o) - ref_o).max() <= TOL[torch.bfloat16]
    assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL[torch.bfloat16]
    plan.close()


def test_bounded_wait_timeout_recovers(vds):
    """A launch whose MMA warp waits for a phase that never completes (test
    hook) ends by itself: the bounded wait expires, the status word says
    WP_ETIMEOUT, and the next launch on the same context is correct.  Both
    the plain and the RoPE kernel."""
    from video_dit_shifted_gb300 import synth
    from oracle import rope as orp
    grid, heads, hd, L = (3, 30, 40, 2, 3, 3), 2, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda", base_seed=17)
    raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
    off, ids = op.layout_tables(*grid, op.REGULAR)
    o = torch.empty((N, heads, hd), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, heads, hd), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, op.REGULAR, heads, hd, L, vds.BF16, "cuda")
    args = (plan, op.REGULAR, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t)
    vds.debug_stall_next(1)
    vds.window_attn(*args, ws)
    assert vds.read_status(ws) == 4                     # WP_ETIMEOUT
    vds.window_attn(*args, ws)
    assert vds.read_status(ws) == 0
    ref_o, ref_t = oa.window_attention(*(raw[n] for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
    assert np.abs(_np(o) - ref_o).max() <= TOL[torch.bfloat16]
    wsr = vds.make_workspace(plan, op.REGULAR, heads, hd, L, vds.BF16, "cuda", rope=True)
    vds.debug_stall_next(1)
    vds.window_attn_rope(*args, wsr)
    assert vds.read_status(wsr) == 4
    vds.window_attn_rope(*args, wsr)
    assert vds.read_status(wsr) == 0
    pv, pt = orp.positions(*grid, op.REGULAR, L)
    ref_o, _ = oa.window_attention(orp.rope(raw["q"], pv), orp.rope(raw["k"], pv), raw["v"],
                                   orp.rope(raw["qt"], pt), orp.rope(raw["kt"], pt), raw["vt"], off, ids)
    assert np.abs(_np(o) - ref_o).max() <= TOL[torch.bfloat16]
    vds.debug_stall_next(0)
    plan.close()


def test_many_heads_and_long_text(vds):
    """40 heads and 1000 text tokens (eight text tiles, the last ragged): the
    work-item decode over heads and the text partial layout at sizes the
    other cases do not reach; three heads checked against the oracle in both
    layouts, the text mean over all windows for those heads."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (2, 30, 40, 1, 2, 2), 40, 128, 1000
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, L, heads, hd, torch.bfloat16, "cuda", base_seed=5)
    raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
    hs = (0, 17, 39)
    for layout in (op.REGULAR, op.SHIFTED):
        o_vid, o_txt, ws = _run(vds, plan, layout, x, heads, hd, L, torch.bfloat16)
        off, ids = op.layout_tables(*grid, layout)
        ref_o, ref_t = oa.window_attention(raw["q"], raw["k"], raw["v"], raw["qt"], raw["kt"], raw["vt"], off, ids,
                                           heads=hs)
        got, got_t = _np(o_vid), _np(o_txt)
        for h in hs:
            assert np.abs(got[:, h] - ref_o[:, h]).max() <= TOL[torch.bfloat16], (layout, h)
            assert np.abs(got_t[:, h] - oa.text_mean(ref_t)[:, h]).max() <= TOL[torch.bfloat16], (layout, h)
        assert not torch.isnan(o_vid).any() and not torch.isnan(o_txt).any()
    plan.close()


def test_two_streams_at_once_match_one_at_a_time(vds):
    """Two layers (different plans, layouts and workspaces) launched on two
    streams at the same time give bit for bit what they give alone: the
    calls share no device state."""
    from video_dit_shifted_gb300 import synth
    cases = [((3, 30, 40, 2, 3, 3), op.REGULAR, 2, 20), ((2, 45, 80, 1, 3, 3), op.SHIFTED, 3, 16)]
    runs = []
    for grid, layout, heads, L in cases:
        plan = vds.Plan(*grid, device="cuda")
        x = synth.attention_inputs(plan.N, L, heads, 128, torch.bfloat16, "cuda", base_seed=layout)
        ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda")
        outs = [(torch.empty((plan.N, heads, 128), dtype=torch.bfloat16, device="cuda"),
                 torch.empty((L, heads, 128), dtype=torch.bfloat16, device="cuda")) for _ in range(2)]
        runs.append((plan, layout, x, ws, outs))
    for plan, layout, x, ws, outs in runs:                 # alone, one after the other
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], *outs[0], ws)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in runs]
    for (plan, layout, x, ws, outs), st in zip(runs, streams):   # both at once
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], *outs[1], ws,
                            stream=st)
    torch.cuda.synchronize()
    for plan, layout, x, ws, outs in runs:
        assert vds.read_status(ws) == 0
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
        plan.close()


def test_text_sum_over_many_windows(vds):
    """The text output is the window-ordered mean of every window's text rows
    (§Text stream).  Many small windows (72 regular, 147 shifted) and three
    text tiles (the last ragged): against the oracle's mean over all windows;
    bit for bit the same on a second call whose workspace was filled with
    garbage first (every per-window text output is written before it is
    read), and on a call on another stream."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (4, 40, 60, 2, 8, 8), 3, 128, 300
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda", base_seed=23)
    raw = [_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")]
    for layout in (op.REGULAR, op.SHIFTED):
        off, ids = op.layout_tables(*grid, layout)
        assert len(off) - 1 >= 72
        o1, t1, ws = _run(vds, plan, layout, x, heads, hd, L, torch.bfloat16)
        ref_o, ref_t = oa.window_attention(*raw, off, ids)
        assert np.abs(_np(o1) - ref_o).max() <= TOL[torch.bfloat16], layout
        assert np.abs(_np(t1) - oa.text_mean(ref_t)).max() <= TOL[torch.bfloat16], layout
        ws.fill_(0xFF)                                   # NaN bit patterns everywhere
        o2, t2 = torch.empty_like(o1), torch.empty_like(t1)
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o2, t2, ws)
        assert vds.read_status(ws) == 0
        assert torch.equal(o1, o2) and torch.equal(t1, t2), layout
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        o3, t3 = torch.empty_like(o1), torch.empty_like(t1)
        with torch.cuda.stream(st):
            vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o3, t3, ws,
                            stream=st)
        torch.cuda.synchronize()
        assert torch.equal(o1, o3) and torch.equal(t1, t3), layout
    plan.close()


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_out_of_range_table_entry_is_reported_not_written(vds, dtype, hd):
    """The plan's device tables live in a caller-owned buffer that must not
    change after the upload.  If an output-row entry is changed to lie past
    the last row anyway, the kernel records WP_EDEVICE in the status word and
    writes nothing for that row; every other row is still right.  The entry
    used here is N + 3 and the output sits inside a larger buffer with guard
    rows, so even an unchecked store would land in memory this test owns."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (3, 30, 40, 2, 3, 3), 2, 20
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    off, ids = op.layout_tables(*grid, op.REGULAR)
    # find the regular layout's id table in the device buffer
    nbytes = plan.device_bytes()
    start = (-plan.dev_buf.data_ptr()) % 256
    tab = plan.dev_buf[start:start + nbytes].view(torch.int32)
    host = tab.cpu().numpy()
    cand = [i for i in np.flatnonzero(host == ids[0]) if i + N <= host.size and np.array_equal(host[i:i + N], ids)]
    # the layout's own table comes first; the fused canonical -> regular
    # permutation table further on holds the same values
    assert len(cand) >= 1
    k = int(off[1]) + 5                                   # a token of window 1
    x = synth.attention_inputs(N, L, heads, hd, dtype, "cuda", base_seed=31)
    big = torch.full((N + 8, heads, hd), 7.0, dtype=dtype, device="cuda")
    o = big[:N]
    t = torch.empty((L, heads, hd), dtype=dtype, device="cuda")
    ws = vds.make_workspace(plan, op.REGULAR, heads, hd, L, code, "cuda")
    tab[cand[0] + k] = N + 3
    try:
        o.fill_(float("nan"))
        vds.window_attn(plan, op.REGULAR, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        assert vds.read_status(ws) == 5                   # WP_EDEVICE
        assert torch.all(big[N:] == 7.0)                  # nothing written past the output
        ref_o, _ = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        got = _np(o)
        missing = int(ids[k])                             # the row that entry should have written
        assert np.all(np.isnan(got[missing]))
        keep = np.ones(N, bool)
        keep[missing] = False
        assert np.abs(got[keep] - ref_o[keep]).max() <= TOL[dtype]
    finally:
        tab[cand[0] + k] = int(ids[k])
    vds.window_attn(plan, op.REGULAR, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
    assert vds.read_status(ws) == 0
    plan.close()


@pytest.mark.parametrize("grid,heads,hd,L", [((21, 68, 120, 4, 3, 3), 24, 128, 256),
                                             ((2, 30, 40, 1, 2, 2), 40, 128, 1000),
                                             ((3, 30, 40, 2, 3, 3), 2, 64, 300)])
def test_text_mean_is_the_ordered_fp32_mean(vds, grid, heads, hd, L):
    """o_txt must be, bit for bit, the window-ordered fp32 sum of the
    per-window text outputs T_w that the attention kernel leaves in the
    workspace, divided by the window count and rounded to bf16 (computed
    here on the host, one window after the other)."""
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, L, heads, hd, torch.bfloat16, "cuda", base_seed=37)
    for layout in (op.REGULAR, op.SHIFTED):
        o_vid, o_txt, ws = _run(vds, plan, layout, x, heads, hd, L, torch.bfloat16)
        nwin = plan.info(layout)["nwin"]
        start = 256                                     # after the status block
        part = ws[start:start + nwin * L * heads * hd * 4].view(torch.float32).view(nwin, L, heads, hd).cpu().numpy()
        acc = np.zeros(part.shape[1:], dtype=np.float32)
        for w in range(nwin):
            acc = acc + part[w]
        want = torch.from_numpy(acc / np.float32(nwin)).to(torch.bfloat16)
        assert torch.equal(o_txt.cpu(), want), layout
    plan.close()


def _random_configs(n, seed=17):
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        grid = (rng.randint(1, 4), rng.randint(4, 40), rng.randint(4, 60),
                rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 4))
        if min(op.window_size(*grid)) < 1:
            continue
        out.append((grid, rng.randint(1, 3), rng.choice([64, 128]), rng.choice([0, 1, 7, 130]),
                    rng.choice([torch.bfloat16, torch.float32])))
    return out


@pytest.mark.parametrize("grid,heads,hd,L,dtype", _random_configs(12))
def test_random_small_configs(vds, grid, heads, hd, L, dtype):
    """Seeded random grids, window counts, head counts, text lengths, head
    dims and dtypes, both layouts, against the oracle (tolerances as above);
    fp32 cases also write their output in a random layout."""
    _check_full(vds, grid, heads, hd, L, dtype)
    if dtype == torch.float32:
        import random
        from video_dit_shifted_gb300 import synth
        out = random.Random(sum(grid)).choice([op.CANONICAL, op.REGULAR, op.SHIFTED])
        plan = vds.Plan(*grid, device="cuda")
        x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda", base_seed=31)
        o = torch.full((plan.N, heads, hd), float("nan"), dtype=dtype, device="cuda")
        t = torch.full((L, heads, hd), float("nan"), dtype=dtype, device="cuda")
        ws = vds.make_workspace(plan, op.SHIFTED, heads, hd, L, vds.FP32, "cuda")
        vds.window_attn(plan, op.SHIFTED, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws,
                        out_layout=out)
        assert vds.read_status(ws) == 0
        off, ids = op.layout_tables(*grid, op.SHIFTED)
        ref_o, _ = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        got = _np(o)
        if out != op.CANONICAL:
            got = got[np.argsort(op.layout_tables(*grid, out)[1])]
        assert np.abs(got - ref_o).max() <= TOL[dtype], out
        plan.close()
