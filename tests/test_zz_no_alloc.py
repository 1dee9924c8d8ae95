"""The allocation-free attention entry point (gpu).

wp_window_attn_static is for callers that cannot allocate device memory at
the moment they run attention (a runtime with its own fixed memory pool that
forbids allocation from plugins, a latency-bound loop that cannot afford the
device synchronisation cudaMalloc may imply).  It takes its scratch from a
fixed array in the library instead of a caller workspace.  These checks call
it through the C ABI and compare it with wp_window_attn on the same inputs,
twice in a row (the shared scratch keeps the previous call's contents), and
check that a request larger than the fixed scratch is refused.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


@pytest.fixture(scope="module")
def vds():
    import __graft_entry__
    __graft_entry__.build()
    import video_dit_shifted_gb300 as m
    return m


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


@pytest.mark.parametrize("dtype,hd", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_static_scratch_matches_workspace_call(vds, dtype, hd):
    from video_dit_shifted_gb300 import synth
    grid, heads, L = (2, 45, 80, 1, 3, 3), 2, 16
    plan = vds.Plan(*grid, device="cuda")
    code = vds.BF16 if dtype == torch.bfloat16 else vds.FP32
    for layout in (vds.REGULAR, vds.SHIFTED):
        x = synth.attention_inputs(plan.N, L, heads, hd, dtype, "cuda", base_seed=7 * layout)
        ref_o = torch.empty((plan.N, heads, hd), dtype=dtype, device="cuda")
        ref_t = torch.empty((L, heads, hd), dtype=dtype, device="cuda")
        ws = vds.make_workspace(plan, layout, heads, hd, L, code, "cuda")
        vds.window_attn(plan, layout, x["q"], x["k"], x["v"], x["qt"], x["kt"], x["vt"], ref_o, ref_t, ws)
        for _ in range(2):
            o = torch.full_like(ref_o, float("nan"))
            t = torch.full_like(ref_t, float("nan"))
            rc = _static(vds, plan, layout, x, o, t)
            assert rc == 0, vds.wp.lib().wp_last_error()
            torch.cuda.synchronize()
            assert (o.float() - ref_o.float()).abs().max().item() <= TOL[dtype]
            assert (t.float() - ref_t.float()).abs().max().item() <= TOL[dtype]
    plan.close()


def test_static_scratch_refuses_oversized_request(vds):
    from video_dit_shifted_gb300 import synth
    # 9 regular windows x 512 text rows x 24 heads x 128 x 4 B of text
    # partials (57 MB): above the fixed scratch.  The inputs have their full
    # sizes, so the call would be well-formed if it were launched.
    plan = vds.Plan(2, 45, 80, 1, 3, 3, device="cuda")
    heads, hd, L = 24, 128, 512
    assert vds.workspace_bytes(plan, vds.REGULAR, heads, hd, L, vds.BF16) > 32 * 1024 * 1024
    x = synth.attention_inputs(plan.N, L, heads, hd, torch.bfloat16, "cuda")
    o = torch.empty((plan.N, heads, hd), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((L, heads, hd), dtype=torch.bfloat16, device="cuda")
    rc = _static(vds, plan, vds.REGULAR, x, o, t)
    assert rc == 2
    assert b"scratch" in vds.wp.lib().wp_last_error()
    plan.close()
