"""Thin ctypes binding of libwp (include/wp.h).

Argument marshalling only: every step of the path runs in libwp's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library is missing, every call raises -- there is no fallback.
"""
import ctypes
import os

import numpy as np
import torch

CANONICAL, REGULAR, SHIFTED = 0, 1, 2
BF16, FP32 = 0, 1
PLAN_HALF_CEIL = 1  # WP_PLAN_HALF_CEIL
STATUS_NAMES = {0: "WP_OK", 1: "WP_EINVAL", 2: "WP_EUNSUPPORTED", 3: "WP_ECUDA",
                4: "WP_ETIMEOUT", 5: "WP_EDEVICE", 6: "WP_ENOTREADY"}

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libwp.so")
_lib = None

_c_int, _c_i64, _c_sz, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
_pi32 = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes); mirrors include/wp.h
SIGNATURES = {
    "wp_plan_create": (_c_int, [_c_int] * 6 + [ctypes.POINTER(_vp)]),
    "wp_plan_create_ex": (_c_int, [_c_int] * 6 + [ctypes.c_uint, ctypes.POINTER(_vp)]),
    "wp_plan_destroy": (None, [_vp]),
    "wp_plan_info": (_c_int, [_vp, _c_int, ctypes.POINTER(_c_i64)] + [ctypes.POINTER(_c_int)] * 5),
    "wp_plan_host_tables": (_c_int, [_vp, _c_int, _pi32, _pi32, _pi32]),
    "wp_plan_device_bytes": (_c_int, [_vp, ctypes.POINTER(_c_sz)]),
    "wp_plan_assign": (_c_int, [_vp, _c_int, _c_int, _pi32, ctypes.POINTER(_c_i64)]),
    "wp_plan_exchange": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_c_i64),
                                  ctypes.POINTER(_c_int), _pi32, _pi32]),
    "wp_plan_upload": (_c_int, [_vp, _vp, _c_sz, _vp]),
    "wp_permute": (_c_int, [_vp, _c_int, _c_int, _vp, _c_i64, _vp, _c_i64, _c_i64, _vp]),
    "wp_rope": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_i64, _vp, _vp, _c_i64,
                         ctypes.c_float, _vp]),
    "wp_attn_workspace_bytes": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                         ctypes.POINTER(_c_sz)]),
    "wp_window_attn": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                _vp, _vp, _vp, _c_i64, _vp, _vp, _vp, _c_i64,
                                _vp, _c_i64, _vp, _vp, _c_sz, ctypes.c_float, _vp]),
    "wp_window_attn_to": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _vp, _vp, _vp, _c_i64, _vp, _vp, _vp, _c_i64,
                                   _vp, _c_i64, _vp, _vp, _c_sz, ctypes.c_float, _vp]),
    "wp_attn_rope_workspace_bytes": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                              ctypes.POINTER(_c_sz)]),
    "wp_window_attn_rope": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _vp, _vp, _vp, _c_i64, _vp, _vp, _vp, _c_i64,
                                     _vp, _c_i64, _vp, _vp, _c_sz, ctypes.c_float, ctypes.c_float, _vp]),
    "wp_window_attn_static": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _vp, _vp, _vp, _c_i64, _vp, _vp, _vp, _c_i64,
                                       _vp, _c_i64, _vp, ctypes.c_float, _vp]),
    "wp_window_attn_fp8": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _vp, _vp, _c_i64, _vp, _c_i64, _vp, _vp, _c_i64, _vp, _c_i64,
                                    ctypes.c_float, ctypes.c_float, _vp, _c_i64, _vp, _vp, _c_sz,
                                    ctypes.c_float, _vp]),
    "wp_quantize_e4m3": (_c_int, [_vp, _c_i64, _c_int, _c_i64, _vp, _c_i64, ctypes.c_float, _vp]),
    "wp_read_status": (_c_int, [_vp, ctypes.POINTER(_c_int), _vp]),
    "wp_debug_stall_next": (_c_int, [_c_int]),
    "wp_last_error": (ctypes.c_char_p, []),
    "wp_abi_version": (_c_int, []),
}


class WpError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__("%s -> %s: %s" % (fn, STATUS_NAMES.get(code, code), msg))
        self.code = code


def lib():
    """The loaded libwp (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libwp.so is not built (run __graft_entry__.build()); "
                               "there is no fallback path")
        l = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _check(fn, code):
    if code != 0:
        raise WpError(fn, code, lib().wp_last_error().decode())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class Plan:
    """Window geometry of one (T, H, W) grid; optionally uploaded to a GPU."""

    def __init__(self, T, H, W, nt, nh, nw, device=None, stream=None, half="floor"):
        """half: how an odd half window is rounded in the shifted layout,
        "floor" (the default) or "ceil" (wp_plan_create_ex in include/wp.h)."""
        if half not in ("floor", "ceil"):
            raise ValueError("half must be 'floor' or 'ceil'")
        h = ctypes.c_void_p()
        flags = PLAN_HALF_CEIL if half == "ceil" else 0
        _check("wp_plan_create_ex", lib().wp_plan_create_ex(T, H, W, nt, nh, nw, flags, ctypes.byref(h)))
        self._h = h
        self.half = half
        self.T, self.H, self.W, self.nt, self.nh, self.nw = T, H, W, nt, nh, nw
        self.N = T * H * W
        self.dev_buf = None
        if device is not None:
            self.upload(device, stream)

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan is closed")
        return self._h

    def info(self, layout):
        n = _c_i64()
        vals = [_c_int() for _ in range(5)]
        _check("wp_plan_info", lib().wp_plan_info(self.handle, layout, ctypes.byref(n),
                                                  *[ctypes.byref(v) for v in vals]))
        nwin, wt, wh, ww, mx = (v.value for v in vals)
        return {"n_tokens": n.value, "nwin": nwin, "window": (wt, wh, ww), "max_tokens": mx}

    def host_tables(self, layout):
        nwin = self.info(layout)["nwin"]
        off = np.zeros(nwin + 1, np.int32)
        ids = np.zeros(self.N, np.int32)
        boxes = np.zeros(nwin * 6, np.int32)
        p = lambda a: a.ctypes.data_as(_pi32)
        _check("wp_plan_host_tables", lib().wp_plan_host_tables(self.handle, layout, p(off), p(ids), p(boxes)))
        return off, ids, boxes.reshape(nwin, 6)

    def assign(self, layout, world):
        """(win_rank[nwin], rank_tokens[world]) of the LPT window -> rank plan."""
        nwin = self.info(layout)["nwin"]
        wr = np.zeros(nwin, np.int32)
        load = np.zeros(world, np.int64)
        _check("wp_plan_assign", lib().wp_plan_assign(self.handle, layout, world, wr.ctypes.data_as(_pi32),
                                                      load.ctypes.data_as(ctypes.POINTER(_c_i64))))
        return wr, load

    def exchange(self, src_layout, dst_layout, world, rank):
        """(counts[world, world], exchange_required, send_rows, recv_pos) of Plan A."""
        C = np.zeros((world, world), np.int64)
        req = _c_int()
        _check("wp_plan_exchange", lib().wp_plan_exchange(
            self.handle, src_layout, dst_layout, world, rank, C.ctypes.data_as(ctypes.POINTER(_c_i64)),
            ctypes.byref(req), None, None))
        send = np.zeros(int(C[rank].sum()), np.int32)
        recv = np.zeros(int(C[:, rank].sum()), np.int32)
        _check("wp_plan_exchange", lib().wp_plan_exchange(
            self.handle, src_layout, dst_layout, world, rank, None, None,
            send.ctypes.data_as(_pi32), recv.ctypes.data_as(_pi32)))
        return C, bool(req.value), send, recv

    def device_bytes(self):
        b = _c_sz()
        _check("wp_plan_device_bytes", lib().wp_plan_device_bytes(self.handle, ctypes.byref(b)))
        return b.value

    def upload(self, device, stream=None):
        device = torch.device(device)
        nbytes = self.device_bytes()
        with torch.cuda.device(device):
            buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
            off = (-buf.data_ptr()) % 256
            view = buf[off:off + nbytes]
            _check("wp_plan_upload", lib().wp_plan_upload(self.handle, _ptr(view), nbytes, _stream_ptr(stream)))
        self.dev_buf = buf
        self.device = device

    def close(self):
        if self._h is not None:
            lib().wp_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def permute(plan, src, dst, src_layout, dst_layout, stream=None):
    """dst[q] = src[row of src_layout holding canonical token ids_dst[q]].

    src, dst: 2-D CUDA tensors [N, ...] (rows may be strided; row bytes are
    the product of the inner dims times the element size)."""
    row_B = src[0].numel() * src.element_size()
    _check("wp_permute", lib().wp_permute(plan.handle, src_layout, dst_layout, _ptr(src),
                                          src.stride(0) * src.element_size(), _ptr(dst),
                                          dst.stride(0) * dst.element_size(), row_B,
                                          _stream_ptr(stream)))
    return dst


def rope(plan, layout, q, k, qt, kt, base=10000.0, stream=None):
    """In-place window-local 3D RoPE of q, k [N, heads, 128] (layout order)
    and qt, kt [L, heads, 128] (see wp_rope in include/wp.h)."""
    N, heads, hd = q.shape
    L = qt.shape[0] if qt is not None else 0
    es = q.element_size()
    if k.stride(0) != q.stride(0) or (L and kt.stride(0) != qt.stride(0)):
        raise ValueError("q and k (and qt and kt) must share one row stride")
    _check("wp_rope", lib().wp_rope(plan.handle, layout, heads, hd, L, _dtype_code(q), _ptr(q), _ptr(k),
                                    q.stride(0) * es, _ptr(qt if L else None), _ptr(kt if L else None),
                                    qt.stride(0) * es if L else 0, float(base), _stream_ptr(stream)))


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def workspace_bytes(plan, layout, heads, head_dim, L, dtype_code):
    b = _c_sz()
    _check("wp_attn_workspace_bytes", lib().wp_attn_workspace_bytes(
        plan.handle, layout, heads, head_dim, L, dtype_code, ctypes.byref(b)))
    return b.value


def rope_workspace_bytes(plan, layout, heads, head_dim, L, dtype_code):
    b = _c_sz()
    _check("wp_attn_rope_workspace_bytes", lib().wp_attn_rope_workspace_bytes(
        plan.handle, layout, heads, head_dim, L, dtype_code, ctypes.byref(b)))
    return b.value


def make_workspace(plan, layout, heads, head_dim, L, dtype_code, device, rope=False):
    n = (rope_workspace_bytes if rope else workspace_bytes)(plan, layout, heads, head_dim, L, dtype_code)
    return torch.empty(n, dtype=torch.uint8, device=device)


def window_attn_rope(plan, layout, q, k, v, qt, kt, vt, o_vid, o_txt, workspace, rope_base=10000.0,
                     scale=0.0, stream=None, out_layout=CANONICAL):
    """Window attention on un-rotated q, k with the window-local RoPE applied
    within the call (wp_window_attn_rope in include/wp.h: k and the text q/k
    rotated once into the workspace, video Q tiles inside the attention
    kernel); q, k, qt, kt are not modified.  Arguments as window_attn;
    workspace from make_workspace(..., rope=True)."""
    N, heads, hd = q.shape
    L = qt.shape[0] if qt is not None else 0
    es = q.element_size()
    if not (k.stride(0) == v.stride(0) == q.stride(0)):
        raise ValueError("q, k, v must share one row stride")
    txt_stride = qt.stride(0) * es if L else 0
    _check("wp_window_attn_rope", lib().wp_window_attn_rope(
        plan.handle, layout, out_layout, heads, hd, L, _dtype_code(q),
        _ptr(q), _ptr(k), _ptr(v), q.stride(0) * es,
        _ptr(qt if L else None), _ptr(kt if L else None), _ptr(vt if L else None), txt_stride,
        _ptr(o_vid), o_vid.stride(0) * es, _ptr(o_txt if L else None),
        _ptr(workspace), workspace.numel(), float(scale), float(rope_base), _stream_ptr(stream)))
    return o_vid, o_txt


def window_attn(plan, layout, q, k, v, qt, kt, vt, o_vid, o_txt, workspace, scale=0.0, stream=None,
                out_layout=CANONICAL):
    """One layer of window attention (wp_window_attn_to in include/wp.h).

    q, k, v: [N, heads, hd] views in `layout` order sharing one row stride;
    qt, kt, vt: [L, heads, hd] sharing one row stride; o_vid [N, heads, hd]
    in `out_layout` order (canonical by default); o_txt [L, heads, hd]
    contiguous."""
    N, heads, hd = q.shape
    L = qt.shape[0] if qt is not None else 0
    es = q.element_size()
    if not (k.stride(0) == v.stride(0) == q.stride(0)):
        raise ValueError("q, k, v must share one row stride")
    txt_stride = qt.stride(0) * es if L else 0
    _check("wp_window_attn_to", lib().wp_window_attn_to(
        plan.handle, layout, out_layout, heads, hd, L, _dtype_code(q),
        _ptr(q), _ptr(k), _ptr(v), q.stride(0) * es,
        _ptr(qt if L else None), _ptr(kt if L else None), _ptr(vt if L else None), txt_stride,
        _ptr(o_vid), o_vid.stride(0) * es, _ptr(o_txt if L else None),
        _ptr(workspace), workspace.numel(), float(scale), _stream_ptr(stream)))
    return o_vid, o_txt


def quantize_e4m3(src, dst, inv_scale, stream=None):
    """dst = e4m3 codes of src * inv_scale (wp_quantize_e4m3 in include/wp.h).

    src: 2-D bf16 CUDA tensor [rows, cols] (row stride may exceed cols);
    dst: 2-D uint8 CUDA tensor of the same shape."""
    if src.dtype != torch.bfloat16 or dst.dtype != torch.uint8 or src.dim() != 2 or dst.shape != src.shape:
        raise TypeError("quantize_e4m3 takes a 2-D bfloat16 src and a uint8 dst of the same shape")
    rows, cols = src.shape
    _check("wp_quantize_e4m3", lib().wp_quantize_e4m3(_ptr(src), rows, cols, src.stride(0) * 2, _ptr(dst),
                                                      dst.stride(0), float(inv_scale), _stream_ptr(stream)))
    return dst


def window_attn_fp8(plan, layout, q8, k8, v, qt8, kt8, vt, q_scale, k_scale, o_vid, o_txt, workspace,
                    scale=0.0, stream=None, out_layout=CANONICAL):
    """Window attention with e4m3 q/k (wp_window_attn_fp8 in include/wp.h).

    q8, k8: uint8 [N, heads, 128] views (e4m3 codes) sharing a row stride;
    v: bf16 [N, heads, 128]; qt8, kt8: uint8 [L, heads, 128]; vt: bf16;
    scores = (q8 * q_scale) . (k8 * k_scale) * scale."""
    N, heads, hd = v.shape
    L = vt.shape[0] if vt is not None else 0
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8 or v.dtype != torch.bfloat16:
        raise TypeError("window_attn_fp8 takes uint8 (e4m3 code) q8/k8 and bfloat16 v")
    if k8.stride(0) != q8.stride(0) or (L and kt8.stride(0) != qt8.stride(0)):
        raise ValueError("q8 and k8 (and qt8 and kt8) must share one row stride")
    _check("wp_window_attn_fp8", lib().wp_window_attn_fp8(
        plan.handle, layout, out_layout, heads, hd, L, _ptr(q8), _ptr(k8), q8.stride(0), _ptr(v), v.stride(0) * 2,
        _ptr(qt8 if L else None), _ptr(kt8 if L else None), qt8.stride(0) if L else 0,
        _ptr(vt if L else None), vt.stride(0) * 2 if L else 0, float(q_scale), float(k_scale),
        _ptr(o_vid), o_vid.stride(0) * 2, _ptr(o_txt if L else None), _ptr(workspace), workspace.numel(),
        float(scale), _stream_ptr(stream)))
    return o_vid, o_txt


def debug_stall_next(launches):
    """Test hook: the next `launches` attention launches time out on purpose
    (wp_debug_stall_next in include/wp.h)."""
    _check("wp_debug_stall_next", lib().wp_debug_stall_next(int(launches)))


def read_status(workspace, stream=None):
    """Device status word of an attention workspace; workspace=None reads the
    fixed scratch of wp_window_attn_static on the current device."""
    st = _c_int()
    _check("wp_read_status", lib().wp_read_status(_ptr(workspace), ctypes.byref(st), _stream_ptr(stream)))
    return st.value
