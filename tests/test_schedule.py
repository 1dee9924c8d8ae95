"""Layer schedule (CPU only).  "Window-Aligned Sequence Parallelism
(SeedVR2)", §Motivation / §Window layouts: the released 32-layer model
alternates layouts and so has 31 inter-layer transitions, derived by
ensure_layout rather than assumed."""
from video_dit_shifted_gb300 import schedule
from video_dit_shifted_gb300.wp import REGULAR, SHIFTED


def test_32_layers_have_31_transitions():
    layouts = schedule.layer_layouts(32)
    assert layouts[:3] == [REGULAR, SHIFTED, REGULAR]
    tr = schedule.transitions(layouts)
    assert len(tr) == 31
    assert tr[0] == (REGULAR, SHIFTED) and tr[1] == (SHIFTED, REGULAR)


def test_ensure_layout_is_derived_not_assumed():
    # a schedule that repeats a layout needs no transition there
    tr = schedule.transitions([REGULAR, REGULAR, SHIFTED, SHIFTED, REGULAR])
    assert tr == [(REGULAR, SHIFTED), (SHIFTED, REGULAR)]
    assert schedule.ensure_layout(SHIFTED, SHIFTED) is None
    assert schedule.transitions([SHIFTED], start=REGULAR) == [(REGULAR, SHIFTED)]


def test_output_layouts_follow_the_next_layer():
    from video_dit_shifted_gb300 import schedule
    lays = schedule.layer_layouts(32)
    outs = schedule.output_layouts(lays)
    assert len(outs) == 32
    assert outs[:-1] == lays[1:]                      # each output in the next layer's order
    assert outs[-1] == schedule.CANONICAL             # the last one back in canonical order
    assert schedule.output_layouts(lays, final=schedule.REGULAR)[-1] == schedule.REGULAR
    assert schedule.output_layouts([schedule.SHIFTED]) == [schedule.CANONICAL]
