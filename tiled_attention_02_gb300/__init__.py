"""tiled_attention_02_gb300 -- Python binding of the tiled exact-attention
C library for GB300 (sm_103a).

Every step of the computation runs in the library's CUDA kernels; this
module only marshals arguments (device pointers of PyTorch tensors, sizes,
the current CUDA stream) into the C ABI declared in ``include/tattn.h`` and
turns a non-OK status into an exception.  There is no CPU or PyTorch
fallback: if the library is missing the calls raise.

Functions mirror the C entry points:

* :func:`attn_fwd` -- ``attn_fwd`` / ``attn_fwd_window`` (O, LSE, optional
  fp32 bias in / logits out, optional causal sliding window)
* :func:`attn_bwd` -- ``attn_bwd`` / ``attn_bwd_window`` / ``attn_bwd_residual``
  (dQ, dK, dV by recomputation; with a bias, the logit gradient in and out)
* :func:`attn_bwd_noalloc` -- ``attn_bwd_noalloc`` (the backward with the
  library's fixed scratch instead of a caller workspace)
* :func:`attn_decode` -- ``attn_decode`` (one new query row per head against
  an N-row K/V cache)
* :func:`attn_bwd_workspace_size`, :func:`attn_decode_workspace_size`,
  :func:`attn_last_device_status`, :func:`attn_status_string`

The ``raw_*`` functions take plain integers (device pointers, sizes, stream
handle) and return the status code, for tests of the C boundary itself.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_DEVICE_CHECK = 5

# Every symbol include/tattn.h declares.
EXPORTED = ("attn_fwd", "attn_fwd_window", "attn_bwd_workspace_size", "attn_bwd",
            "attn_bwd_window", "attn_bwd_residual", "attn_bwd_noalloc", "attn_decode_workspace_size", "attn_decode",
            "attn_status_string",
            "attn_last_device_status", "attn_version", "attn_debug_fwd_timeout")


def _header_define(name: str) -> int:
    """An integer #define of include/tattn.h, read from the header the library
    is compiled against (one source for the value, no copy of it here)."""
    import re
    path = os.path.join(os.path.dirname(_HERE), "include", "tattn.h")
    with open(path) as f:
        m = re.search(r"^#define\s+" + name + r"\s+(\d+)\s*$", f.read(), flags=re.M)
    if not m:
        raise RuntimeError(f"{name} not found in {path}")
    return int(m.group(1))


# Size of the fixed device scratch attn_bwd_noalloc uses.
ATTN_BWD_NOALLOC_SCRATCH_BYTES = _header_define("ATTN_BWD_NOALLOC_SCRATCH_BYTES")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"tattn CUDA library not built: {LIB_PATH} is missing "
                                   "(run tiled_attention_02_gb300.build())")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]
            L.attn_fwd.restype = i
            L.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]
            L.attn_fwd_window.restype = i
            L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i]
            L.attn_bwd_workspace_size.restype = sz
            L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                   sz, vp]
            L.attn_bwd.restype = i
            L.attn_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                          i, vp, sz, vp]
            L.attn_bwd_window.restype = i
            L.attn_bwd_residual.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i,
                                            i, i, i, f, i, vp, sz, vp]
            L.attn_bwd_residual.restype = i
            L.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                           f, i, vp]
            L.attn_bwd_noalloc.restype = i
            L.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
            L.attn_decode_workspace_size.restype = sz
            L.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
            L.attn_decode.restype = i
            L.attn_debug_fwd_timeout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i,
                                                 ctypes.c_ulonglong, vp]
            L.attn_debug_fwd_timeout.restype = i
            L.attn_status_string.argtypes = [i]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_last_device_status.argtypes = [vp]
            L.attn_last_device_status.restype = i
            L.attn_version.argtypes = []
            L.attn_version.restype = i
            _lib = L
    return _lib


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(t, name, dtype, shape):
    """Type, shape and layout of one tensor argument (None passes)."""
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_all(specs, device):
    """Checks every (tensor, name, dtype, shape) of a call, inputs and
    caller-given outputs alike, before anything reaches the library: first
    type, shape and layout, then that each lives on `device` (a CUDA
    device).  A wrong output buffer would otherwise be written out of
    bounds by the kernels."""
    for t, name, dt, shp in specs:
        _check(t, name, dt, shp)
    for t, name, _, _ in specs:
        if t is not None and (not t.is_cuda or t.device != device):
            raise TypeError(f"{name} must be a CUDA tensor on {device}, got {t.device}")


def raw_attn_fwd(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, scale, causal, emit, stream) -> int:
    """The C entry point with raw integer pointers; returns the status code."""
    return lib().attn_fwd(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, ctypes.c_float(scale),
                          int(causal), emit, stream)


def raw_attn_fwd_window(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, scale, window, emit,
                       stream) -> int:
    return lib().attn_fwd_window(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, ctypes.c_float(scale),
                                 int(window), emit, stream)


def raw_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal, ws,
                 ws_bytes, stream) -> int:
    return lib().attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D,
                          ctypes.c_float(scale), int(causal), ws, ws_bytes, stream)


def raw_attn_bwd_residual(q, k, v, o, lse, do, bias, grad_in, dq, dk, dv, grad_out, B, Hq, Hkv,
                          N, D, scale, causal, ws, ws_bytes, stream) -> int:
    return lib().attn_bwd_residual(q, k, v, o, lse, do, bias, grad_in, dq, dk, dv, grad_out, B,
                                   Hq, Hkv, N, D, ctypes.c_float(scale), int(causal), ws,
                                   ws_bytes, stream)


def raw_attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D, scale, window, ws,
                        ws_bytes, stream) -> int:
    return lib().attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D,
                                 ctypes.c_float(scale), int(window), ws, ws_bytes, stream)


def attn_fwd(q, k, v, bias=None, *, scale: float | None = None, causal: bool = False,
             o=None, lse=None, emit_logits=None, want_lse: bool = True, stream=None,
             window: int | None = None):
    """Exact attention forward through the C ABI.

    q [B,Hq,N,D], k/v [B,Hkv,N,D] bf16 CUDA tensors; bias (optional) fp32
    [B,Hq,N,N]; emit_logits (optional) fp32 [B,Hq,N,N] output buffer, which
    may be ``bias`` itself.  ``window`` (with causal=True): causal sliding
    window of that many keys (attn_fwd_window).  Returns ``(o, lse)`` (lse
    is None when ``want_lse`` is False and no ``lse`` buffer is given).
    """
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_all(((q, "q", torch.bfloat16, (B, Hq, N, D)),
                (k, "k", torch.bfloat16, (B, Hkv, N, D)),
                (v, "v", torch.bfloat16, (B, Hkv, N, D)),
                (bias, "bias", torch.float32, (B, Hq, N, N)),
                (emit_logits, "emit_logits", torch.float32, (B, Hq, N, N)),
                (o, "o", torch.bfloat16, (B, Hq, N, D)),
                (lse, "lse", torch.float32, (B, Hq, N))), q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if window is not None:
        if not causal:
            raise ValueError("a sliding window needs causal=True")
        st = raw_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(o), _ptr(lse), B,
                                 Hq, Hkv, N, D, scale, window, _ptr(emit_logits),
                                 _stream_handle(stream))
    else:
        st = raw_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(o), _ptr(lse), B, Hq, Hkv,
                          N, D, scale, causal, _ptr(emit_logits), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return o, lse


def _bwd_specs(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D):
    import torch
    bf = torch.bfloat16
    return ((q, "q", bf, (B, Hq, N, D)), (k, "k", bf, (B, Hkv, N, D)),
            (v, "v", bf, (B, Hkv, N, D)), (o, "o", bf, (B, Hq, N, D)),
            (lse, "lse", torch.float32, (B, Hq, N)), (do, "do", bf, (B, Hq, N, D)),
            (dq, "dq", bf, (B, Hq, N, D)), (dk, "dk", bf, (B, Hkv, N, D)),
            (dv, "dv", bf, (B, Hkv, N, D)))


def raw_attn_debug_fwd_timeout(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, causal, wait_limit_ns,
                               stream) -> int:
    """Test hook: the forward with block 0's first K load left out and every
    pipeline wait bounded by `wait_limit_ns` (see include/tattn.h)."""
    return lib().attn_debug_fwd_timeout(q, k, v, o, lse, B, Hq, Hkv, N, D, ctypes.c_float(scale),
                                        int(causal), int(wait_limit_ns), stream)


def attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, N: int, D: int) -> int:
    return int(lib().attn_bwd_workspace_size(B, Hq, Hkv, N, D))


def attn_bwd(q, k, v, o, lse, do, *, scale: float | None = None, causal: bool = False,
             dq=None, dk=None, dv=None, workspace=None, stream=None,
             window: int | None = None, bias=None, grad_in=None, grad_out=None):
    """Backward by recomputation through the C ABI; returns (dq, dk, dv).

    Block attention residual (attn_bwd_residual): ``bias`` is the forward's
    fp32 [B,Hq,N,N] logit bias, ``grad_in`` the gradient arriving at this
    layer's logits from the next layer, and ``grad_out`` (may be grad_in)
    receives this layer's total logit gradient."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    residual = bias is not None or grad_in is not None or grad_out is not None
    if residual and window is not None:
        raise ValueError("the residual backward takes no window")
    if workspace is not None and (not isinstance(workspace, torch.Tensor)
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous tensor")
    _check_all(_bwd_specs(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D)
               + ((bias, "bias", torch.float32, (B, Hq, N, N)),
                  (grad_in, "grad_in", torch.float32, (B, Hq, N, N)),
                  (grad_out, "grad_out", torch.float32, (B, Hq, N, N)),
                  (workspace, "workspace", None if workspace is None else workspace.dtype,
                   None if workspace is None else tuple(workspace.shape))), q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_bwd_workspace_size(B, Hq, Hkv, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if residual:
        st = raw_attn_bwd_residual(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                   _ptr(bias), _ptr(grad_in), _ptr(dq), _ptr(dk), _ptr(dv),
                                   _ptr(grad_out), B, Hq, Hkv, N, D, scale, causal,
                                   _ptr(workspace), ws_bytes, _stream_handle(stream))
    elif window is not None:
        if not causal:
            raise ValueError("a sliding window needs causal=True")
        st = raw_attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, N, D, scale, window,
                                 _ptr(workspace), ws_bytes, _stream_handle(stream))
    else:
        st = raw_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, Hq, Hkv, N, D, scale, causal, _ptr(workspace),
                          ws_bytes, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def raw_attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal,
                         stream) -> int:
    return lib().attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D,
                                  ctypes.c_float(scale), int(causal), stream)


def attn_bwd_noalloc(q, k, v, o, lse, do, *, scale: float | None = None, causal: bool = False,
                     dq=None, dk=None, dv=None, stream=None):
    """Backward through the allocation-free C entry point: the library's own
    fixed device scratch replaces the workspace (for callers that cannot
    allocate device memory).  Output tensors are allocated here only when
    not given.  Returns (dq, dk, dv)."""
    import torch
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_all(_bwd_specs(q, k, v, o, lse, do, dq, dk, dv, B, Hq, Hkv, N, D), q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = raw_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                              _ptr(dk), _ptr(dv), B, Hq, Hkv, N, D, scale, causal,
                              _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_noalloc")
    return dq, dk, dv


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, N: int, D: int) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, N, D))


def raw_attn_decode(q, k, v, o, lse, B, Hq, Hkv, N, D, scale, ws, ws_bytes, stream) -> int:
    return lib().attn_decode(q, k, v, o, lse, B, Hq, Hkv, N, D, ctypes.c_float(scale), ws,
                             ws_bytes, stream)


def attn_decode(q, k, v, *, scale: float | None = None, o=None, lse=None, want_lse: bool = True,
                workspace=None, stream=None):
    """Decode step through the C ABI: q [B,Hq,D] (one new row per query head)
    against the cache k/v [B,Hkv,N,D].  Returns (o [B,Hq,D], lse [B,Hq])."""
    import torch
    B, Hq, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if workspace is not None and (not isinstance(workspace, torch.Tensor)
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous tensor")
    _check_all(((q, "q", torch.bfloat16, (B, Hq, D)),
                (k, "k", torch.bfloat16, (B, Hkv, N, D)),
                (v, "v", torch.bfloat16, (B, Hkv, N, D)),
                (o, "o", torch.bfloat16, (B, Hq, D)),
                (lse, "lse", torch.float32, (B, Hq)),
                (workspace, "workspace", None if workspace is None else workspace.dtype,
                 None if workspace is None else tuple(workspace.shape))), q.device)
    o = torch.empty_like(q) if o is None else o
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = attn_decode_workspace_size(B, Hq, Hkv, N, D)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = raw_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, D, scale,
                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                         _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode")
    return o, lse


def attn_last_device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device status word."""
    return int(lib().attn_last_device_status(_stream_handle(stream)))
