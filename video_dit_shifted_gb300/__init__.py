"""Shifted-window video attention for GB300 (sm_103a).

The hot path of NaDiT/SeedVR2-style video DiTs ("Window-Aligned Sequence
Parallelism (SeedVR2)"): a host window planner, the regular <-> shifted row
re-layout, and window attention over [video window ; replicated text] with
the per-window text outputs averaged over the window count.  The compute
runs in libwp.so (include/wp.h); ``wp`` is its ctypes binding.
"""
from . import wp  # noqa: F401
from .wp import (BF16, CANONICAL, FP32, REGULAR, SHIFTED, Plan, debug_stall_next,  # noqa: F401
                 make_workspace, permute, quantize_e4m3, read_status, rope, rope_workspace_bytes, window_attn,
                 window_attn_fp8, window_attn_rope, workspace_bytes)
