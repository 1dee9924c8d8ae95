"""Layer schedule: which layout each layer runs in, and where the re-layout
(wp_permute) happens.

"Window-Aligned Sequence Parallelism (SeedVR2)", §Motivation and §Window
layouts: regular and shifted layouts alternate layer by layer, and the
transitions are derived from the actual schedule with
ensure_layout(current, required) rather than assumed from layer % 2.  The
page leaves open which layout the first layer uses; layer 0 is regular here.
"""
from .wp import CANONICAL, REGULAR, SHIFTED


def layer_layouts(num_layers, first=REGULAR):
    other = SHIFTED if first == REGULAR else REGULAR
    return [first if l % 2 == 0 else other for l in range(num_layers)]


def ensure_layout(current, required):
    """The (src, dst) re-layout to issue before a layer, or None."""
    return None if current == required else (current, required)


def transitions(layouts, start=None):
    """Re-layouts a schedule needs: one per change of layout between layers
    (plus one into the first layer if the data starts elsewhere)."""
    out, cur = [], layouts[0] if start is None else start
    for req in layouts:
        t = ensure_layout(cur, req)
        if t is not None:
            out.append(t)
        cur = req
    return out


def output_layouts(layouts, final=CANONICAL):
    """Where each layer's video attention output goes when it is written
    straight into the next layer's order (wp_window_attn_to's out_layout):
    the next layer's layout, and `final` (canonical order by default) after
    the last layer.  Written this way, a schedule needs no re-layout of the
    attention output between layers (§Plan A redistribution: at SP=1 a
    transition is a local permutation, here folded into the epilogue)."""
    return [layouts[l + 1] if l + 1 < len(layouts) else final for l in range(len(layouts))]
