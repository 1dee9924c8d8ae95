"""The alternating layer schedule on the GPU (gpu).

"Window-Aligned Sequence Parallelism (SeedVR2)", §Motivation and §Window
layouts: layers alternate the regular and the shifted layout, and the packed
q/k/v rows are re-laid out between layers.  Run through the public calls
(wp_window_attn, wp_permute) as a model would: every even layer must give the
regular layer's result bit for bit, every odd layer the shifted layer's, both
must match the oracle (max abs error <= 2e-2, bf16), and the re-layouts must
bring the rows back to where they started.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import permute as opm
from oracle import plan as op

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


def test_six_layers_alternate_and_match_the_oracle(vds):
    from video_dit_shifted_gb300 import schedule, synth
    # 2 x 2 x 2 regular and 3 x 3 x 3 shifted windows of up to 3x15x27 tokens
    grid, heads, hd, L = (6, 30, 54, 2, 3, 3), 3, 128, 48
    plan = vds.Plan(*grid, device="cuda")
    N = plan.N
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, "cuda", base_seed=11)
    start = x["vid_buf"].clone()                     # rows in regular order
    bufs = [x["vid_buf"], torch.empty_like(x["vid_buf"])]
    txt = x["txt_buf"]
    layouts = schedule.layer_layouts(6)
    assert len(schedule.transitions(layouts)) == 5
    ws = {l: vds.make_workspace(plan, l, heads, hd, L, vds.BF16, "cuda") for l in (op.REGULAR, op.SHIFTED)}
    o_vid = torch.full((6, N, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_txt = torch.full((6, L, heads, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    cur = 0
    for l, lay in enumerate(layouts):
        b = bufs[cur]
        vds.window_attn(plan, lay, b[:, 0], b[:, 1], b[:, 2], txt[:, 0], txt[:, 1], txt[:, 2], o_vid[l], o_txt[l],
                        ws[lay])
        if l + 1 < len(layouts):
            vds.permute(plan, bufs[cur].view(N, -1), bufs[1 - cur].view(N, -1), lay, layouts[l + 1])
            cur = 1 - cur
    torch.cuda.synchronize()
    for w in ws.values():
        assert vds.read_status(w) == 0
    for l in range(2, 6):
        assert torch.equal(o_vid[l], o_vid[l - 2]) and torch.equal(o_txt[l], o_txt[l - 2]), l

    # the rows are now in shifted order; one more re-layout restores the start exactly
    back = torch.empty_like(start)
    vds.permute(plan, bufs[cur].view(N, -1), back.view(N, -1), layouts[-1], op.REGULAR)
    assert torch.equal(back, start)

    host = _np(start)                                 # [N, 3, heads, hd], regular order
    ttxt = [_np(txt[:, i]) for i in range(3)]
    ids = {l: op.layout_tables(*grid, l)[1] for l in (op.REGULAR, op.SHIFTED)}
    for l, lay in enumerate(layouts[:2]):
        rows = host if lay == op.REGULAR else opm.permute_rows(host, ids[op.REGULAR], ids[op.SHIFTED])
        off, lay_ids = op.layout_tables(*grid, lay)
        ref_o, ref_t = oa.window_attention(rows[:, 0], rows[:, 1], rows[:, 2], *ttxt, off, lay_ids)
        assert np.abs(_np(o_vid[l]) - ref_o).max() <= TOL, lay
        assert np.abs(_np(o_txt[l]) - oa.text_mean(ref_t)).max() <= TOL, lay
    plan.close()
