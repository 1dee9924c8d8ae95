"""wp_rope (window-local 3D RoPE, in place) against the oracle (gpu).

Tolerances.  bf16: 2e-2 max abs, as for attention.  fp32: 1e-4 max abs.
Basis of the fp32 figure: the kernel forms each angle as float(pos) *
theta_i in fp32, with theta_i = base^(-2i/42) rounded once to fp32 on the
host, so the angle carries at most 2 * 2^-24 * |pos * theta_i| of error
(the oracle's angles are float64), and sincosf adds a few ulp; a rotated
value x0 c - x1 s is then off by at most (|x0| + |x1|) * (angle error +
2^-22) plus the rounding of two products and a sum.  On these grids
|pos * theta_i| <= 39 (the canonical layout's widest axis) and |x| < 6 for
N(0,1) draws of this size, which bounds the error near 4e-5.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import plan as op
from oracle import rope as orp

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("L", [0, 5])
def test_rope_matches_oracle(vds, dtype, L):
    from video_dit_shifted_gb300 import synth
    grid, heads = (3, 30, 40, 2, 3, 3), 3
    plan = vds.Plan(*grid, device="cuda")
    for layout in (op.REGULAR, op.SHIFTED, op.CANONICAL):
        x = synth.attention_inputs(plan.N, max(L, 1), heads, 128, dtype, "cuda", base_seed=layout)
        qt, kt = (x["qt"], x["kt"]) if L else (None, None)
        before = {n: _np(x[n]) for n in ("q", "k", "qt", "kt")}
        vds.rope(plan, layout, x["q"], x["k"], qt, kt)
        torch.cuda.synchronize()
        pv, pt = orp.positions(*grid, layout, L)
        for n, pos in (("q", pv), ("k", pv)) + ((("qt", pt), ("kt", pt)) if L else ()):
            want = orp.rope(before[n], pos)
            assert np.abs(_np(x[n]) - want).max() <= TOL[dtype], (layout, n)
    plan.close()


def test_rope_then_attention(vds):
    """RoPE in the layer's layout followed by window attention equals the
    oracle's rotated attention."""
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (2, 45, 80, 1, 3, 3), 2, 16
    plan = vds.Plan(*grid, device="cuda")
    for layout in (op.REGULAR, op.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, 128, torch.bfloat16, "cuda", base_seed=5 * layout)
        raw = {n: _np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")}
        vds.rope(plan, layout, x["q"], x["k"], x["qt"], x["kt"])
        o = torch.empty((plan.N, heads, 128), dtype=torch.bfloat16, device="cuda")
        t = torch.empty((L, heads, 128), dtype=torch.bfloat16, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, 128, L, vds.BF16, "cuda")
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
        pv, pt = orp.positions(*grid, layout, L)
        off, ids = op.layout_tables(*grid, layout)
        ref_o, ref_t = oa.window_attention(orp.rope(raw["q"], pv), orp.rope(raw["k"], pv), raw["v"],
                                           orp.rope(raw["qt"], pt), orp.rope(raw["kt"], pt), raw["vt"], off, ids)
        assert np.abs(_np(o) - ref_o).max() <= 2e-2
        assert np.abs(_np(t) - oa.text_mean(ref_t)).max() <= 2e-2
    plan.close()


def test_rope_1080p_sampled_rows(vds):
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (21, 68, 120, 4, 3, 3), 24, 256
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, L, heads, 128, torch.bfloat16, "cuda")
    rows = np.random.default_rng(0).choice(plan.N, 2048, replace=False)
    idx = torch.from_numpy(rows).cuda()
    before_q, before_qt = _np(x["q"][idx]), _np(x["qt"])
    vds.rope(plan, op.SHIFTED, x["q"], x["k"], x["qt"], x["kt"])
    torch.cuda.synchronize()
    pv, pt = orp.positions(*grid, op.SHIFTED, L)
    assert np.abs(_np(x["q"][idx]) - orp.rope(before_q, pv[rows])).max() <= 2e-2
    assert np.abs(_np(x["qt"]) - orp.rope(before_qt, pt)).max() <= 2e-2
    plan.close()


def test_rope_rejects_head_dim_64(vds):
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    q = torch.zeros((plan.N, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vds.wp.WpError) as e:
        vds.rope(plan, op.REGULAR, q, q.clone(), None, None)
    assert e.value.code == 2
    plan.close()


def _random_cases(n, seed=29):
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        grid = (rng.randint(1, 5), rng.randint(2, 40), rng.randint(2, 40),
                rng.randint(1, 4), rng.randint(1, 4), rng.randint(1, 4))
        if min(op.window_size(*grid)) < 1:
            continue
        out.append((grid, rng.randint(1, 3), rng.choice([0, 3, 20]),
                    rng.choice([torch.bfloat16, torch.float32]), rng.choice([op.REGULAR, op.SHIFTED])))
    return out


@pytest.mark.parametrize("grid,heads,L,dtype,layout", _random_cases(8))
def test_random_grids(vds, grid, heads, L, dtype, layout):
    """Seeded random grids, window counts, head counts, text lengths (<= 20,
    so positions stay within the range of the fp32 basis above), dtypes and
    layouts, against the oracle's rotation."""
    from video_dit_shifted_gb300 import synth
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, max(L, 1), heads, 128, dtype, "cuda", base_seed=sum(grid))
    qt, kt = (x["qt"][:L], x["kt"][:L]) if L else (None, None)
    before = {n: _np(x[n]) for n in ("q", "k", "qt", "kt")}
    vds.rope(plan, layout, x["q"], x["k"], qt, kt)
    torch.cuda.synchronize()
    pv, pt = orp.positions(*grid, layout, L)
    assert np.abs(_np(x["q"]) - orp.rope(before["q"], pv)).max() <= TOL[dtype]
    assert np.abs(_np(x["k"]) - orp.rope(before["k"], pv)).max() <= TOL[dtype]
    if L:
        assert np.abs(_np(x["qt"][:L]) - orp.rope(before["qt"][:L], pt)).max() <= TOL[dtype]
        assert np.abs(_np(x["kt"][:L]) - orp.rope(before["kt"][:L], pt)).max() <= TOL[dtype]
    plan.close()
