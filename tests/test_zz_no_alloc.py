"""The allocation-free attention entry point (gpu).

wp_window_attn_static is for callers that cannot allocate device memory at
the moment they run attention (a runtime with its own fixed memory pool that
forbids allocation from plugins, a latency-bound loop that cannot afford the
device synchronisation cudaMalloc may imply).  It takes its scratch from a
fixed array in the library instead of a caller workspace.  These checks call
it through the C ABI:

* it runs the same kernels as wp_window_attn on the same inputs, so its
  outputs must equal the workspace call's bit for bit, on two calls in a row
  (the shared scratch keeps the previous call's contents), on the small PR1
  grid in both dtypes and on the 720p-like video grid at full size;
* on the PR1 grid it matches the oracle (bf16 2e-2, fp32 1e-4);
* after the first call on the device (the set-up, which may load the
  library's device code), later calls leave the device's free memory as it
  was;
* a bounded wait that expires inside it is reported by wp_read_status with a
  NULL workspace, and the next call is correct;
* a request larger than the fixed scratch is refused before any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import plan as op

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


def _static(vds, plan, layout, x, o_vid, o_txt):
    lib = vds.wp.lib()
    q, k, v, qt, kt, vt = (x[n] for n in ("q", "k", "v", "qt", "kt", "vt"))
    N, heads, hd = q.shape
    L = qt.shape[0]
    es = q.element_size()
    code = vds.BF16 if q.dtype == torch.bfloat16 else vds.FP32
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.wp_window_attn_static(
        plan.handle, layout, heads, hd, L, code, p(q), p(k), p(v), q.stride(0) * es,
        p(qt), p(kt), p(vt), qt.stride(0) * es, p(o_vid), o_vid.stride(0) * es, p(o_txt),
        ctypes.c_float(0.0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _static_status(vds):
    st = ctypes.c_int(-1)
    rc = vds.wp.lib().wp_read_status(None, ctypes.byref(st),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, vds.wp.lib().wp_last_error()
    return st.value


def _workspace_call(vds, plan, layout, x):
    q = x["q"]
    N, heads, hd = q.shape
    L = x["qt"].shape[0]
    code = vds.BF16 if q.dtype == torch.bfloat16 else vds.FP32
    o = torch.empty((N, heads, hd), dtype=q.dtype, device="cuda")
    t = torch.empty((L, heads, hd), dtype=q.dtype, device="cuda")
    ws = vds.make_workspace(plan, layout, heads, hd, L, code, "cuda")
    vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], o, t, ws)
    assert vds.read_status(ws) == 0
    return o, t


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_static_scratch_matches_workspace_call_and_oracle(vds, dtype, hd):
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (2, 45, 80, 1, 3, 3), 2, 16
    plan = vds.Plan(*grid, device="cuda")
    for layout in (vds.REGULAR, vds.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda", base_seed=7 * layout)
        ref_o, ref_t = _workspace_call(vds, plan, layout, x)
        outs = [(torch.full_like(ref_o, float("nan")), torch.full_like(ref_t, float("nan"))) for _ in range(2)]
        for o, t in outs:                          # two calls in a row
            rc = _static(vds, plan, layout, x, o, t)
            assert rc == 0, vds.wp.lib().wp_last_error()
            assert _static_status(vds) == 0
            assert torch.equal(o, ref_o) and torch.equal(t, ref_t), layout
        off, ids = op.layout_tables(*grid, layout)
        want_o, want_t = oa.window_attention(*(_np(x[n]) for n in ("q", "k", "v", "qt", "kt", "vt")), off, ids)
        assert np.abs(_np(outs[1][0]) - want_o).max() <= TOL[dtype]
        assert np.abs(_np(outs[1][1]) - oa.text_mean(want_t)).max() <= TOL[dtype]
    plan.close()


def test_static_scratch_full_size_layer_allocates_nothing(vds):
    """The 720p-like video grid (T=21, 45x80, 24 heads x 128) with 16 text
    tokens, in both layouts: its scratch (36 or 64 windows of text outputs,
    up to 12.6 MB) fits the fixed array.  Bit-equal to the workspace call on
    two calls in a row; once the set-up call has run, the device's free
    memory is the same before and after every later call."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (21, 45, 80, 4, 3, 3), 24, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, L, heads, hd, torch.bfloat16, "cuda")
    for layout in (vds.REGULAR, vds.SHIFTED):
        ref_o, ref_t = _workspace_call(vds, plan, layout, x)
        outs = [(torch.empty_like(ref_o), torch.empty_like(ref_t)) for _ in range(3)]
        assert _static(vds, plan, layout, x, *outs[0]) == 0       # set-up (first call on the device)
        torch.cuda.synchronize()
        for o, t in outs[1:]:
            free0 = torch.cuda.mem_get_info()[0]
            assert _static(vds, plan, layout, x, o, t) == 0, vds.wp.lib().wp_last_error()
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0
            assert _static_status(vds) == 0
        for o, t in outs:
            assert torch.equal(o, ref_o) and torch.equal(t, ref_t), layout
    plan.close()


def test_static_scratch_reports_a_timeout(vds):
    """The test hook makes one launch's bounded wait expire: the static
    call still returns (the fault is on the device), wp_read_status(NULL)
    reports WP_ETIMEOUT, and the next static call is correct again."""
    from video_dit_shifted_gb300 import synth
    grid, heads, hd, L = (3, 30, 40, 2, 3, 3), 2, 128, 16
    plan = vds.Plan(*grid, device="cuda")
    x = synth.attention_inputs(plan.N, L, heads, hd, torch.bfloat16, "cuda", base_seed=17)
    ref_o, ref_t = _workspace_call(vds, plan, vds.REGULAR, x)
    o, t = torch.empty_like(ref_o), torch.empty_like(ref_t)
    vds.debug_stall_next(1)
    assert _static(vds, plan, vds.REGULAR, x, o, t) == 0
    assert _static_status(vds) == 4                                 # WP_ETIMEOUT
    vds.debug_stall_next(0)
    assert _static(vds, plan, vds.REGULAR, x, o, t) == 0
    assert _static_status(vds) == 0
    assert torch.equal(o, ref_o) and torch.equal(t, ref_t)
    plan.close()


@pytest.mark.parametrize("dtype,L", [(torch.bfloat16, 4096), (torch.float32, 512)])
def test_static_scratch_refuses_oversized_request(vds, dtype, L):
    from video_dit_shifted_gb300 import synth
    # per-window text outputs [9, L, 24, 128] fp32: 453 MB (bf16, L = 4096)
    # and 57 MB (fp32, L = 512), both above the fixed scratch.  The inputs
    # have their full sizes, so the call would be well-formed if it were
    # launched.
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    heads, hd = 24, 128
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    assert vds.workspace_bytes(plan, vds.REGULAR, heads, hd, L, code) > 32 * 1024 * 1024
    x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda")
    o = torch.empty((plan.N, heads, hd), dtype=dtype, device="cuda")
    t = torch.empty((L, heads, hd), dtype=dtype, device="cuda")
    rc = _static(vds, plan, vds.REGULAR, x, o, t)
    assert rc == 2
    assert b"scratch" in vds.wp.lib().wp_last_error()
    plan.close()
