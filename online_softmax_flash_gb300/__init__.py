"""Python binding of libosf (include/osf.h): same entry-point names, argument marshalling only.

Every step of attention and softmax runs in libosf's CUDA kernels.  PyTorch supplies device
memory and the current CUDA stream.  There is no fallback: if libosf.so is missing or a
tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "OSF_OK", "OSF_ERR_INVALID", "OSF_ERR_UNSUPPORTED", "OSF_ERR_CUDA", "OSF_ERR_TIMEOUT",
    "OSF_ERR_WORKSPACE", "OSF_F32", "OSF_BF16", "OsfError", "lib", "library_path",
    "osf_status_string", "osf_version", "osf_sm_count", "osf_attn_fwd", "osf_attn_fwd_gqa",
    "osf_attn_workspace_bytes", "osf_attn_decode_gqa", "osf_attn_decode_workspace_bytes",
    "osf_softmax_rows", "osf_softmax_workspace_bytes", "osf_device_status", "osf_launch_count",
    "solve", "osf_attn_fwd_gqa_ex", "osf_softmax_rows_ex", "osf_softmax_ex_workspace_bytes",
    "osf_attn_bwd_gqa", "osf_attn_bwd_workspace_bytes", "osf_selftest_bounded_wait", "OSF_MASK_NONE", "OSF_MASK_TOP_LEFT", "OSF_MASK_BOTTOM_RIGHT",
    "osf_attn_fwd_gqa_host", "osf_attn_host_buffer_bytes",
]

OSF_OK, OSF_ERR_INVALID, OSF_ERR_UNSUPPORTED, OSF_ERR_CUDA, OSF_ERR_TIMEOUT, OSF_ERR_WORKSPACE = range(6)
OSF_F32, OSF_BF16 = 0, 1

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libosf.so")
_lib = None

_vp, _sz, _i, _ll, _f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
_SIGS = {
    "osf_status_string": (ctypes.c_char_p, [_i]),
    "osf_version": (_i, []),
    "osf_sm_count": (_i, []),
    "osf_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "osf_attn_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "osf_attn_workspace_bytes": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "osf_attn_fwd_gqa_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "osf_attn_host_buffer_bytes": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "osf_attn_fwd_gqa_ex": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _i, _f, _vp, _vp, _sz, _vp]),
    "osf_attn_decode_gqa": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _i, _vp, _sz, _vp]),
    "osf_attn_decode_workspace_bytes": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "osf_softmax_rows": (_i, [_vp, _vp, _ll, _ll, _vp, _sz, _vp]),
    "osf_softmax_rows_ex": (_i, [_vp, _vp, _i, _i, _ll, _ll, _ll, _ll, _f, _ll, _vp, _sz, _vp]),
    "osf_softmax_ex_workspace_bytes": (_i, [_ll, _ll, ctypes.POINTER(_sz)]),
    "osf_attn_bwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f,
                              _vp, _sz, _vp]),
    "osf_attn_bwd_workspace_bytes": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "osf_selftest_bounded_wait": (_i, [ctypes.c_ulonglong, _vp]),
    "osf_softmax_workspace_bytes": (_i, [_ll, _ll, ctypes.POINTER(_sz)]),
    "osf_device_status": (_i, [_vp]),
    "osf_launch_count": (ctypes.c_ulonglong, []),
}


class OsfError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {osf_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libosf.so (built by ``_build.build()``); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"libosf.so not found at {library_path}: build it first "
                               "(online_softmax_flash_gb300._build.build())")
        l = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(status: int, where: str) -> None:
    if status != OSF_OK:
        raise OsfError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _need_cuda(*ts, contiguous: bool = True) -> None:
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libosf works on CUDA tensors only (no CPU path)")
        if contiguous and t is not None and not t.is_contiguous():
            raise ValueError("libosf expects contiguous row-major tensors")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return OSF_F32
    if t.dtype == torch.bfloat16:
        return OSF_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def osf_status_string(status: int) -> str:
    return lib().osf_status_string(int(status)).decode()


def osf_version() -> int:
    return lib().osf_version()


def osf_sm_count() -> int:
    return lib().osf_sm_count()


def osf_attn_fwd(Q, K, V, out, M: int, N: int, d: int) -> None:
    """out[M, d] = softmax(Q K^T / sqrt(d)) V for float32 Q[M, d], K[N, d], V[N, d]."""
    _need_cuda(Q, K, V, out)
    _check(lib().osf_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(out), M, N, d, _stream(Q.device)),
           "osf_attn_fwd")


def solve(Q, K, V, output, M: int, N: int, d: int) -> None:
    """The pages' ``solve(Q, K, V, output, M, N, d)``: osf_attn_fwd, then wait for it."""
    osf_attn_fwd(Q, K, V, output, M, N, d)
    torch.cuda.current_stream(Q.device).synchronize()


def osf_attn_workspace_bytes(dtype: int, B, Hq, Hkv, Sq, Sk, D) -> int:
    n = _sz(0)
    _check(lib().osf_attn_workspace_bytes(dtype, B, Hq, Hkv, Sq, Sk, D, ctypes.byref(n)),
           "osf_attn_workspace_bytes")
    return n.value


def _workspace(nbytes: int, dev, workspace):
    if nbytes == 0:
        return workspace
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return workspace


def osf_attn_fwd_gqa(q, k, v, out=None, causal: bool = False, scale: float | None = None,
                     lse=None, workspace=None):
    """Grouped-query attention on [B, H, S, D] tensors; returns ``out`` (allocated if None)."""
    _need_cuda(q, k, v, out, lse)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    ws_n = osf_attn_workspace_bytes(dt, B, Hq, Hkv, Sq, Sk, D)
    ws = _workspace(ws_n, q.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().osf_attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), dt, B, Hq, Hkv, Sq, Sk, D,
                                  int(bool(causal)), 0.0 if scale is None else float(scale),
                                  _ptr(lse), _ptr(ws), ws_bytes, _stream(q.device)),
           "osf_attn_fwd_gqa")
    return out


def osf_attn_host_buffer_bytes(dtype: int, B, Hq, Hkv, Sq, Sk, D, causal: bool = False) -> int:
    n = _sz(0)
    _check(lib().osf_attn_host_buffer_bytes(dtype, B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), ctypes.byref(n)),
           "osf_attn_host_buffer_bytes")
    return n.value


def osf_attn_fwd_gqa_host(q, k, v, out=None, causal: bool = False, scale: float | None = None,
                          device_buffer=None, device=None):
    """osf_attn_fwd_gqa on host (CPU) tensors: the library copies them in, runs the attention and
    copies O back, overlapping the copies with the computation; ``out`` (a host tensor, pinned if
    ``q`` is) is allocated if None.  ``device_buffer``: a CUDA uint8 tensor of at least
    osf_attn_host_buffer_bytes bytes, allocated on ``device`` (default: the current device) if
    None.  Returns ``out``, which holds the result once the device's current stream has reached
    the end of the call (synchronise it before reading)."""
    for t in (q, k, v, out):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("osf_attn_fwd_gqa_host takes contiguous host tensors")
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    n = osf_attn_host_buffer_bytes(dt, B, Hq, Hkv, Sq, Sk, D, causal)
    if device_buffer is None:
        device_buffer = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    _need_cuda(device_buffer)
    nb = device_buffer.numel() * device_buffer.element_size()
    with torch.cuda.device(device_buffer.device):
        _check(lib().osf_attn_fwd_gqa_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), dt, B, Hq, Hkv, Sq, Sk, D,
                                           int(bool(causal)), 0.0 if scale is None else float(scale),
                                           _ptr(device_buffer), nb, _stream(device_buffer.device)),
               "osf_attn_fwd_gqa_host")
    return out


OSF_MASK_NONE, OSF_MASK_TOP_LEFT, OSF_MASK_BOTTOM_RIGHT = 0, 1, 2
_MASKS = {"none": OSF_MASK_NONE, "top_left": OSF_MASK_TOP_LEFT, "bottom_right": OSF_MASK_BOTTOM_RIGHT}


def osf_attn_fwd_gqa_ex(q, k, v, out=None, mask="none", scale: float | None = None, lse=None,
                        workspace=None):
    """Grouped-query attention on logical [B, H, S, D] views with any strides (the last
    dimension contiguous), e.g. ``x.transpose(1, 2)`` of a [B, S, H, D] tensor; ``mask`` is
    "none", "top_left", "bottom_right" (or an OSF_MASK_* code).  ``out`` defaults to a
    contiguous [B, Hq, Sq, D] tensor; ``lse`` must be a contiguous float32 [B, Hq, Sq]."""
    _need_cuda(q, k, v, out, lse, contiguous=False)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=q.dtype, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 4 or (t.shape[3] > 1 and t.stride(3) != 1):
            raise ValueError(f"{name} must be a 4-D [B, H, S, D] view with a contiguous last dimension")
    if lse is not None and not lse.is_contiguous():
        raise ValueError("lse must be contiguous")
    st = (ctypes.c_longlong * 12)(*(int(t.stride(i)) for t in (q, k, v, out) for i in range(3)))
    m = _MASKS[mask] if isinstance(mask, str) else int(mask)
    ws_n = osf_attn_workspace_bytes(dt, B, Hq, Hkv, Sq, Sk, D)
    ws = _workspace(ws_n, q.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().osf_attn_fwd_gqa_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), dt, B, Hq, Hkv, Sq, Sk, D,
                                     ctypes.cast(st, ctypes.c_void_p), m,
                                     0.0 if scale is None else float(scale), _ptr(lse), _ptr(ws), ws_bytes,
                                     _stream(q.device)),
           "osf_attn_fwd_gqa_ex")
    return out


def osf_attn_bwd_workspace_bytes(dtype: int, B, Hq, Hkv, Sq, Sk, D) -> int:
    n = _sz(0)
    _check(lib().osf_attn_bwd_workspace_bytes(dtype, B, Hq, Hkv, Sq, Sk, D, ctypes.byref(n)),
           "osf_attn_bwd_workspace_bytes")
    return n.value


def osf_attn_bwd_gqa(q, k, v, o, dout, lse, dq=None, dk=None, dv=None, mask="none",
                     scale: float | None = None, workspace=None):
    """Gradients (dq, dk, dv) of GQA attention on contiguous [B, H, S, D] tensors, given the
    forward output ``o``, its log-sum-exp ``lse`` and the gradient ``dout`` of the loss with
    respect to ``o``; ``mask`` and ``scale`` as in the forward call."""
    _need_cuda(q, k, v, o, dout, lse, dq, dk, dv)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = _MASKS[mask] if isinstance(mask, str) else int(mask)
    ws_n = osf_attn_bwd_workspace_bytes(dt, B, Hq, Hkv, Sq, Sk, D)
    ws = _workspace(ws_n, q.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().osf_attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), dt, B, Hq, Hkv, Sq, Sk, D, m, 0.0 if scale is None else float(scale),
                                  _ptr(ws), ws_bytes, _stream(q.device)),
           "osf_attn_bwd_gqa")
    return dq, dk, dv


def osf_attn_decode_workspace_bytes(dtype: int, B, Hq, Hkv, Sk, D, num_splits: int = 0) -> int:
    n = _sz(0)
    _check(lib().osf_attn_decode_workspace_bytes(dtype, B, Hq, Hkv, Sk, D, num_splits, ctypes.byref(n)),
           "osf_attn_decode_workspace_bytes")
    return n.value


def osf_attn_decode_gqa(q, k, v, out=None, scale: float | None = None, lse=None,
                        num_splits: int = 0, workspace=None):
    """Sq == 1 attention with an explicit split count over the keys."""
    _need_cuda(q, k, v, out, lse)
    B, Hq, Sq, D = q.shape
    if Sq != 1:
        raise ValueError("osf_attn_decode_gqa expects q of shape [B, Hq, 1, D]")
    Hkv, Sk = k.shape[1], k.shape[2]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    ws_n = osf_attn_decode_workspace_bytes(dt, B, Hq, Hkv, Sk, D, num_splits)
    ws = _workspace(ws_n, q.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().osf_attn_decode_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), dt, B, Hq, Hkv, Sk, D,
                                     0.0 if scale is None else float(scale), _ptr(lse),
                                     int(num_splits), _ptr(ws), ws_bytes, _stream(q.device)),
           "osf_attn_decode_gqa")
    return out


def osf_softmax_workspace_bytes(rows: int, T: int) -> int:
    n = _sz(0)
    _check(lib().osf_softmax_workspace_bytes(rows, T, ctypes.byref(n)), "osf_softmax_workspace_bytes")
    return n.value


def osf_softmax_rows(x, z=None, workspace=None):
    """Row softmax of a float32 [rows, T] (or 1-D [T]) tensor; ``z is x`` runs in place."""
    _need_cuda(x, z)
    if x.dtype != torch.float32:
        raise ValueError("osf_softmax_rows takes float32")
    T = x.shape[-1] if x.dim() > 0 else 1
    rows = x.numel() // T if T else 0
    if z is None:
        z = torch.empty_like(x)
    ws_n = osf_softmax_workspace_bytes(rows, T)
    ws = _workspace(ws_n, x.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().osf_softmax_rows(_ptr(x), _ptr(z), rows, T, _ptr(ws), ws_bytes, _stream(x.device)),
           "osf_softmax_rows")
    return z


def osf_softmax_ex_workspace_bytes(rows: int, T: int) -> int:
    n = _sz(0)
    _check(lib().osf_softmax_ex_workspace_bytes(rows, T, ctypes.byref(n)), "osf_softmax_ex_workspace_bytes")
    return n.value


def osf_softmax_rows_ex(x, z=None, out_dtype=None, scale: float = 1.0, causal_period: int = 0, workspace=None):
    """Row softmax of ``scale * x`` for a float32 or bfloat16 [rows, T] view whose rows may be
    strided (``x.stride(1) == 1``); ``causal_period`` P > 0 keeps columns ``0 .. r % P`` of row
    r.  ``z`` (default: a new contiguous tensor of ``out_dtype``, else ``x.dtype``) may be ``x``."""
    _need_cuda(x, z, contiguous=False)
    if x.dim() != 2:
        raise ValueError("osf_softmax_rows_ex takes a 2-D [rows, T] tensor")
    rows, T = x.shape
    if z is None:
        z = torch.empty((rows, T), dtype=out_dtype or x.dtype, device=x.device)
    for name, t in (("x", x), ("z", z)):
        if t.shape != (rows, T) or (T > 1 and t.stride(1) != 1):
            raise ValueError(f"{name} must be [rows, T] with contiguous rows")
    ws_n = osf_softmax_ex_workspace_bytes(rows, T)
    ws = _workspace(ws_n, x.device, workspace)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    xs = x.stride(0) if rows > 1 else T
    zs = z.stride(0) if rows > 1 else T
    _check(lib().osf_softmax_rows_ex(_ptr(x), _ptr(z), _dtype_code(x), _dtype_code(z), rows, T, xs, zs,
                                     float(scale), int(causal_period), _ptr(ws), ws_bytes, _stream(x.device)),
           "osf_softmax_rows_ex")
    return z


def osf_selftest_bounded_wait(limit_ns: int = 1_000_000) -> int:
    """Run the bounded-wait self-test kernel; returns the launch status (the timeout itself is
    reported by osf_device_status())."""
    return lib().osf_selftest_bounded_wait(int(limit_ns), _stream(torch.cuda.current_device()))


def osf_launch_count() -> int:
    """Kernels launched by libosf so far in this process."""
    return lib().osf_launch_count()


def osf_device_status() -> int:
    """Synchronise the current stream and return (and clear) the device status word."""
    return lib().osf_device_status(_stream(torch.cuda.current_device()))
