"""The e4m3 attention variant (gpu).

* wp_quantize_e4m3 gives the oracle's codes bit for bit (an integer
  decision: both sides take it from the same float32 product x * inv_scale).
* wp_window_attn_fp8, fed the oracle's codes, matches the oracle's attention
  on the decoded q/k (max abs error <= 2e-2, the bf16 tolerance: the kernel's
  arithmetic after the quantisation is the bf16 path's).
* Against exact attention on the unquantised q/k the error is the e4m3
  rounding's (3 mantissa bits: each q, k element carries up to 2^-4
  relative error); it is measured here and bounded by FP8_TOL, a figure
  taken from these measurements, not from the pages.  Measured on a GB300:
  0.029 (3x30x40 grid, windows of 1200-2430 tokens, L = 300), 0.081 (the
  same grid without text), 0.044 (the PR1 grid, L = 16), 0.118 (segments
  of 53 keys, where a softmax averages fewer scores and their rounding
  shows more).
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import plan as op
from oracle import quant as oq

pytestmark = pytest.mark.gpu

TOL = 2e-2          # against the oracle on the decoded q/k
FP8_TOL = 0.15      # against the oracle on the unquantised q/k (measured, above)
INV = 64.0          # power of two: decoded value = code / 64 exactly


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _codes(x):
    """Oracle codes of a bf16 tensor, as a uint8 CUDA tensor of its shape."""
    c = oq.quantize(x.float().cpu().numpy(), INV)
    return torch.from_numpy(c).cuda()


def test_quantize_matches_oracle_bit_for_bit(vds):
    g = torch.Generator(device="cuda").manual_seed(3)
    rows, cols = 3000, 384
    wide = torch.randn((rows, cols + 64), device="cuda", generator=g)
    wide[:, :64] *= 1e-3                               # subnormal codes after scaling
    wide[:, 64:96] *= 40.0                             # saturation
    wide[0, :16] = torch.tensor([1.0625, 1.1875, -1.0625, 0.0, -0.0, 7.0, 7.5, 6.75,
                                 1e-7, -1e-7, 448.0, 500.0, -500.0, 2.0 ** -15, 3 * 2.0 ** -16, 1.0])
    src = wide.to(torch.bfloat16)[:, :cols]            # strided rows
    dst_buf = torch.full((rows, cols + 32), 0x55, dtype=torch.uint8, device="cuda")
    dst = dst_buf[:, 16:16 + cols]
    vds.quantize_e4m3(src, dst, 1.0)
    torch.cuda.synchronize()
    want = oq.quantize(src.float().cpu().numpy(), 1.0)
    assert np.array_equal(dst.cpu().numpy(), want)
    vds.quantize_e4m3(src, dst, INV)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), oq.quantize(src.float().cpu().numpy(), INV))
    assert torch.all(dst_buf[:, :16] == 0x55) and torch.all(dst_buf[:, 16 + cols:] == 0x55)


def _run_fp8(vds, plan, layout, x, codes, heads, L, out_layout=op.CANONICAL):
    N = plan.N
    o = torch.full((N, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    t = torch.full((L, heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda")
    vds.window_attn_fp8(plan, layout, codes["q"], codes["k"], x["v"], codes["qt"], codes["kt"], x["vt"],
                        1.0 / INV, 1.0 / INV, o, t, ws, out_layout=out_layout)
    assert vds.read_status(ws) == 0
    return o, t


def _packed_codes(x, names=("q", "k")):
    """Oracle codes of q and k packed as [N, 2, heads, 128] (and text the same)."""
    out = {}
    for pre, n in (("", x["q"].shape[0]), ("t", x["qt"].shape[0])):
        buf = torch.empty((n, 2) + tuple(x["q"].shape[1:]), dtype=torch.uint8, device="cuda")
        buf[:, 0] = _codes(x["q" + pre])
        buf[:, 1] = _codes(x["k" + pre])
        out["q" + pre], out["k" + pre] = buf[:, 0], buf[:, 1]
    return out


@pytest.mark.parametrize("grid,heads,L", [((3, 30, 40, 2, 3, 3), 2, 300), ((2, 45, 80, 1, 3, 3), 3, 16),
                                          ((2, 45, 80, 1, 9, 16), 2, 3), ((3, 30, 40, 2, 3, 3), 2, 0)])
def test_fp8_attention_matches_oracle(vds, grid, heads, L):
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    errs = []
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, 128, torch.bfloat16, "cuda", base_seed=4 * layout)
        codes = _packed_codes(x)
        off, ids = op.layout_tables(*grid, layout)
        dq = {n: oq.decode(codes[n].cpu().numpy()) / INV for n in ("q", "k", "qt", "kt")}
        ref_o, ref_t = oa.window_attention(dq["q"], dq["k"], _np(x["v"]), dq["qt"], dq["kt"], _np(x["vt"]),
                                           off, ids)
        exact_o, exact_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        other = op.SHIFTED if layout == op.REGULAR else op.REGULAR
        for out in (op.CANONICAL, layout, other):
            o, t = _run_fp8(vds, plan, layout, x, codes, heads, L, out)
            got = _np(o)
            if out != op.CANONICAL:        # output row r holds canonical token ids_out[r]
                got = got[np.argsort(op.layout_tables(*grid, out)[1])]
            assert np.abs(got - ref_o).max() <= TOL, (layout, out)
            err = np.abs(got - exact_o).max()
            if L:
                assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL, (layout, out)
                err = max(err, np.abs(_np(t) - oa.text_mean(exact_t)).max())
            errs.append(err)
    print("e4m3 attention, max abs error against the unquantised oracle:", max(errs))
    assert max(errs) <= FP8_TOL
    plan.close()


def test_fp8_1080p_sampled(vds):
    """The 1080p-like layer at full size in both layouts, launched as the
    bench launches it: every head of a few windows against the oracle on the
    decoded q/k, and the quantiser's codes of 4096 sampled rows of q and k
    (all heads) against the oracle's bit for bit."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (21, 68, 120, 4, 3, 3), 24, 256
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, 128, torch.bfloat16, "cuda")
    qk = torch.empty((N, 2, heads, 128), dtype=torch.uint8, device="cuda")
    qkt = torch.empty((L, 2, heads, 128), dtype=torch.uint8, device="cuda")
    for i, n in enumerate(("q", "k")):
        vds.quantize_e4m3(x[n].reshape(N, heads * 128), qk[:, i].reshape(N, heads * 128), INV)
        vds.quantize_e4m3(x[n + "t"].reshape(L, heads * 128), qkt[:, i].reshape(L, heads * 128), INV)
    torch.cuda.synchronize()
    sample = torch.from_numpy(np.random.default_rng(4).choice(N, 4096, replace=False)).cuda()
    for i, n in enumerate(("q", "k")):
        want = oq.quantize(x[n][sample].float().cpu().numpy(), INV)
        assert np.array_equal(qk[sample, i].cpu().numpy(), want), n
    codes = {"q": qk[:, 0], "k": qk[:, 1], "qt": qkt[:, 0], "kt": qkt[:, 1]}
    rng = np.random.default_rng(5)
    for layout in (op.REGULAR, op.SHIFTED):
        o, t = _run_fp8(vds, plan, layout, x, codes, heads, L)
        assert not torch.isnan(o).any() and not torch.isnan(t).any()
        off, ids = op.layout_tables(*grid, layout)
        sizes = np.diff(off)
        wins = sorted({0, len(sizes) - 1, int(sizes.argmin()), int(rng.integers(len(sizes)))})
        rows = np.concatenate([np.arange(off[w], off[w + 1]) for w in wins])
        sel = torch.from_numpy(rows).cuda()
        dq = lambda c: oq.decode(c.cpu().numpy()) / INV
        sub_off = np.concatenate([[0], np.cumsum(sizes[wins])])
        ref_o, _ = oa.window_attention(dq(codes["q"][sel]), dq(codes["k"][sel]), _np(x["v"][sel]), dq(codes["qt"]),
                                       dq(codes["kt"]), _np(x["vt"]), sub_off, np.arange(rows.size))
        got = _np(o[torch.from_numpy(ids[rows]).cuda()])
        assert np.abs(got - ref_o).max() <= TOL, layout
        exact_o, _ = oa.window_attention(_np(x["q"][sel]), _np(x["k"][sel]), _np(x["v"][sel]), _np(x["qt"]),
                                         _np(x["kt"]), _np(x["vt"]), sub_off, np.arange(rows.size))
        err = np.abs(got - exact_o).max()
        print("e4m3 attention, 1080p-like layer %d, max abs error against the unquantised oracle: %.4f"
              % (layout, err))
        assert err <= FP8_TOL, layout
    plan.close()


def test_fp8_rejections(vds):
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    N, L = plan.N, 16
    x = synth.attention_inputs(N, L, 2, 64, torch.bfloat16, "cuda")
    c = {n: torch.zeros(x[n].shape, dtype=torch.uint8, device="cuda") for n in ("q", "k", "qt", "kt")}
    o = torch.empty((N, 2, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, 2, 64), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, op.REGULAR, 2, 64, L, vds.BF16, "cuda")
    with pytest.raises(vds.wp.WpError) as e:                       # head_dim 64
        vds.window_attn_fp8(plan, op.REGULAR, c["q"], c["k"], x["v"], c["qt"], c["kt"], x["vt"], 1.0, 1.0, o, t, ws)
    assert e.value.code == 2
    x = synth.attention_inputs(N, L, 2, 128, torch.bfloat16, "cuda")
    c = {n: torch.zeros(x[n].shape, dtype=torch.uint8, device="cuda") for n in ("q", "k", "qt", "kt")}
    o = torch.empty((N, 2, 128), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, 2, 128), dtype=torch.bfloat16, device="cuda")
    ws = vds.make_workspace(plan, op.REGULAR, 2, 128, L, vds.BF16, "cuda")
    for qs in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(vds.wp.WpError) as e:
            vds.window_attn_fp8(plan, op.REGULAR, c["q"], c["k"], x["v"], c["qt"], c["kt"], x["vt"], qs, 1.0, o, t, ws)
        assert e.value.code == 1
    src = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vds.wp.WpError) as e:                       # cols not a multiple of 16
        vds.quantize_e4m3(src, torch.zeros((4, 24), dtype=torch.uint8, device="cuda"), 1.0)
    assert e.value.code == 2
    plan.close()


def _random_cases(n, seed=41):
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        grid = (rng.randint(1, 4), rng.randint(4, 40), rng.randint(4, 60),
                rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 4))
        if min(op.window_size(*grid)) < 1:
            continue
        out.append((grid, rng.randint(1, 3), rng.choice([0, 1, 7, 130])))
    return out


@pytest.mark.parametrize("grid,heads,L", _random_cases(4))
def test_fp8_random_configs(vds, grid, heads, L):
    """Seeded random grids, window counts, head counts and text lengths: the
    e4m3 call fed the oracle's codes against the oracle on the decoded q/k."""
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, 128, torch.bfloat16, "cuda", base_seed=sum(grid) + layout)
        codes = _packed_codes(x)
        off, ids = op.layout_tables(*grid, layout)
        dq = {n: oq.decode(codes[n].cpu().numpy()) / INV for n in ("q", "k", "qt", "kt")}
        ref_o, ref_t = oa.window_attention(dq["q"], dq["k"], _np(x["v"]), dq["qt"], dq["kt"], _np(x["vt"]), off, ids)
        o, t = _run_fp8(vds, plan, layout, x, codes, heads, L)
        assert np.abs(_np(o) - ref_o).max() <= TOL, layout
        if L:
            assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= TOL, layout
    plan.close()
