"""The C ABI library loads, exports what include/wp.h declares, and rejects
bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def wp():
    import __graft_entry__
    __graft_entry__.build()
    from video_dit_shifted_gb300 import wp as _wp
    return _wp


def _declared():
    text = open(os.path.join(ROOT, "include", "wp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wp_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(wp):
    names = _declared()
    assert len(names) >= 12
    lib = wp.lib()
    for n in names:
        assert hasattr(lib, n), n
    # and the binding's signature table covers the header exactly
    assert sorted(wp.SIGNATURES) == names


def test_abi_version(wp):
    assert wp.lib().wp_abi_version() == 1


def test_plan_create_rejects_bad_arguments(wp):
    lib = wp.lib()
    h = ctypes.c_void_p()
    for args in [(0, 45, 80, 1, 3, 3), (2, 45, 80, 0, 3, 3), (2, -1, 80, 1, 3, 3),
                 (2000, 2000, 2000, 1, 1, 1),      # N >= 2^31
                 (1, 1, 100000, 1, 1, 1)]:         # round(H*scale) = 0
        rc = lib.wp_plan_create(*args, ctypes.byref(h))
        assert rc == 1, args
        assert lib.wp_last_error()
    assert lib.wp_plan_create(2, 45, 80, 1, 3, 3, None) == 1


def test_calls_validate_before_cuda(wp):
    lib = wp.lib()
    plan = wp.Plan(2, 45, 80, 1, 3, 3)             # host only, not uploaded
    vp = ctypes.c_void_p
    # permute: bad layouts, null pointers, unaligned rows, overlap
    assert lib.wp_permute(plan.handle, 3, 1, vp(16), 16, vp(1 << 40), 16, 16, None) == 1
    assert lib.wp_permute(plan.handle, 1, 2, None, 16, vp(1 << 40), 16, 16, None) == 1
    assert lib.wp_permute(plan.handle, 1, 2, vp(16), 24, vp(1 << 40), 24, 24, None) == 2
    assert lib.wp_permute(plan.handle, 1, 2, vp(8), 16, vp(1 << 40), 16, 16, None) == 2
    assert lib.wp_permute(plan.handle, 1, 2, vp(1 << 20), 32, vp((1 << 20) + 64), 32, 32, None) == 1
    # not uploaded -> WP_ENOTREADY, still without any launch
    assert lib.wp_permute(plan.handle, 1, 2, vp(1 << 20), 32, vp(1 << 40), 32, 32, None) in (3, 6)
    # attention: bad layout, head_dim, null pointers, small workspace
    args = lambda layout, hd, ws_bytes: (plan.handle, layout, 2, hd, 16, 0, vp(256), vp(512), vp(768), 8192,
                                         vp(1024), vp(1280), vp(1536), 8192, vp(4096), 8192, vp(2048),
                                         vp(1 << 30), ws_bytes, ctypes.c_float(0.0), None)
    assert lib.wp_window_attn(*args(0, 128, 1 << 30)) == 1
    assert lib.wp_window_attn(*args(1, 96, 1 << 30)) == 2
    assert lib.wp_window_attn(*args(1, 128, 64)) == 1
    # degenerate head and text counts
    hargs = lambda heads, L: (plan.handle, 1, heads, 128, L, 0, vp(256), vp(512), vp(768), 8192, vp(1024),
                              vp(1280), vp(1536), 8192, vp(4096), 8192, vp(2048), vp(1 << 30), 1 << 30,
                              ctypes.c_float(0.0), None)
    for heads, L in [(0, 16), (-1, 16), (1 << 20, 16), (2, -1)]:
        assert lib.wp_window_attn(*hargs(heads, L)) == 1, (heads, L)
        assert lib.wp_last_error()
    size = ctypes.c_size_t()
    # status block, per-window text outputs [9, 16, 2, 128] fp32 (either dtype)
    assert lib.wp_attn_workspace_bytes(plan.handle, 1, 2, 128, 16, 0, ctypes.byref(size)) == 0
    assert size.value == 256 + 9 * 16 * 2 * 128 * 4
    fsize = ctypes.c_size_t()
    assert lib.wp_attn_workspace_bytes(plan.handle, 1, 2, 128, 16, 1, ctypes.byref(fsize)) == 0
    assert fsize.value == size.value
    # RoPE attention: the workspace adds the rotated text q and k (bf16), then
    # (1024-byte aligned) the rotated video k [N, heads, 128] bf16, N = 2*45*80
    rsize = ctypes.c_size_t()
    assert lib.wp_attn_rope_workspace_bytes(plan.handle, 1, 2, 128, 16, 0, ctypes.byref(rsize)) == 0
    krot = (size.value + 2 * 16 * 2 * 128 * 2 + 1023) // 1024 * 1024
    assert rsize.value == krot + 7200 * 2 * 128 * 2
    rargs = lambda layout, hd, dtype, ws_bytes, base: (
        plan.handle, layout, 0, 2, hd, 16, dtype, vp(256), vp(512), vp(768), 8192, vp(1024), vp(1280), vp(1536),
        8192, vp(4096), 8192, vp(2048), vp(1 << 30), ws_bytes, ctypes.c_float(0.0), ctypes.c_float(base), None)
    assert lib.wp_window_attn_rope(*rargs(1, 128, 0, 1 << 30, 1.0)) == 1       # rope_base <= 1
    assert lib.wp_window_attn_rope(*rargs(1, 128, 1, 1 << 30, 1e4)) == 2       # fp32
    assert lib.wp_window_attn_rope(*rargs(1, 64, 0, 1 << 30, 1e4)) == 2        # head_dim 64
    assert lib.wp_window_attn_rope(*rargs(1, 128, 0, size.value, 1e4)) == 1    # no room for the rotated text
    assert lib.wp_window_attn_rope(*rargs(1, 128, 0, rsize.value, 1e4)) in (3, 6)  # not uploaded
    plan.close()


def test_e4m3_calls_validate_before_cuda(wp):
    lib = wp.lib()
    vp = ctypes.c_void_p
    f = ctypes.c_float
    # wp_quantize_e4m3(src, rows, cols, src_stride, dst, dst_stride, inv_scale, stream)
    assert lib.wp_quantize_e4m3(None, 4, 32, 64, vp(4096), 32, f(1.0), None) == 1          # NULL src
    assert lib.wp_quantize_e4m3(vp(4096), -1, 32, 64, vp(8192), 32, f(1.0), None) == 1     # negative rows
    assert lib.wp_quantize_e4m3(vp(4096), 4, 24, 48, vp(8192), 32, f(1.0), None) == 2      # cols % 16
    assert lib.wp_quantize_e4m3(vp(4104), 4, 32, 64, vp(8192), 32, f(1.0), None) == 2      # unaligned src
    assert lib.wp_quantize_e4m3(vp(4096), 4, 32, 48, vp(8192), 32, f(1.0), None) == 2      # stride < row
    for bad in (0.0, -2.0, float("inf"), float("nan")):
        assert lib.wp_quantize_e4m3(vp(4096), 4, 32, 64, vp(8192), 32, f(bad), None) == 1
    assert lib.wp_quantize_e4m3(vp(4096), 0, 32, 64, vp(8192), 32, f(1.0), None) == 0      # nothing to do
    # wp_window_attn_fp8: head_dim, scales, strides, workspace, then the plan
    plan = wp.Plan(2, 45, 80, 1, 3, 3)
    size = ctypes.c_size_t()
    assert lib.wp_attn_workspace_bytes(plan.handle, 1, 2, 128, 16, 0, ctypes.byref(size)) == 0
    args = lambda hd, qs, qk_stride, v_stride, ws_bytes: (
        plan.handle, 1, 0, 2, hd, 16, vp(256), vp(512), qk_stride, vp(1024), v_stride, vp(2048), vp(2304),
        qk_stride, vp(4096), v_stride, f(qs), f(1.0), vp(8192), 512, vp(16384), vp(1 << 30), ws_bytes, f(0.0), None)
    assert lib.wp_window_attn_fp8(*args(64, 1.0, 256, 512, size.value)) == 2      # head_dim 64
    assert lib.wp_window_attn_fp8(*args(128, 0.0, 256, 512, size.value)) == 1     # scale
    assert lib.wp_window_attn_fp8(*args(128, 1.0, 240, 512, size.value)) == 2     # q/k stride < row (256 B)
    assert lib.wp_window_attn_fp8(*args(128, 1.0, 256, 256, size.value)) == 2     # v stride < row (512 B)
    assert lib.wp_window_attn_fp8(*args(128, 1.0, 256, 512, 64)) == 1             # workspace too small
    assert lib.wp_window_attn_fp8(*args(128, 1.0, 256, 512, size.value)) in (3, 6)  # not uploaded
    plan.close()


def test_debug_stall_hook_validates(wp):
    lib = wp.lib()
    assert lib.wp_debug_stall_next(-1) == 1
    assert lib.wp_debug_stall_next(0) == 0


def test_plan_info(wp):
    plan = wp.Plan(21, 68, 120, 4, 3, 3)
    assert plan.info(wp.REGULAR) == {"n_tokens": 171360, "nwin": 100, "window": (6, 15, 27),
                                     "max_tokens": 2430}
    assert plan.info(wp.SHIFTED)["nwin"] == 120
    assert plan.info(wp.CANONICAL)["nwin"] == 1
    plan.close()
