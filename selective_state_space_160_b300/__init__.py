"""Mamba selective scan (S6 forward / backward, Mamba-2 SSD chunked forward) for
NVIDIA B300 (sm_103a).

Every step of the computation runs in libmsc.so (hand-written CUDA behind the C
ABI declared in include/msc.h).  This module only marshals arguments: it takes
torch CUDA tensors, allocates outputs and workspace with torch, and passes raw
device pointers plus the current CUDA stream to the library.  There is no CPU
fallback: if the library is missing or a tensor is not on the GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "load_library", "library_path",
    "msc_selective_scan_fwd", "msc_selective_scan_bwd", "msc_ssd_chunked_fwd", "msc_ssd_chunked_bwd",
    "msc_selective_state_update", "msc_ssd_chunked_bwd_workspace_size",
    "msc_causal_conv1d_fwd", "msc_causal_conv1d_update", "msc_selective_scan_fwd_ex",
    "msc_selective_scan_fwd_conv", "msc_causal_conv1d_bwd", "msc_selective_scan_fwd_host",
    "msc_selective_scan_fwd_train", "msc_selective_scan_bwd_ckpt", "msc_selective_scan_ckpt_size",
    "MSC_DISC_EULER", "MSC_DISC_ZOH", "MSC_DISC_TRAPEZOID",
    "msc_selective_scan_fwd_workspace_size", "msc_selective_scan_bwd_workspace_size",
    "msc_ssd_chunked_fwd_workspace_size", "msc_check_device_status", "msc_status_string",
    "msc_last_error", "MscError", "MSC_F32", "MSC_BF16",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libmsc.so")
_lock = threading.Lock()
_lib = None

MSC_OK, MSC_ERR_INVALID_ARG, MSC_ERR_UNSUPPORTED, MSC_ERR_CUDA, MSC_ERR_TIMEOUT, MSC_ERR_WORKSPACE = range(6)
MSC_F32, MSC_BF16 = 0, 1
MSC_DISC_EULER, MSC_DISC_ZOH, MSC_DISC_TRAPEZOID = 0, 1, 2

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/msc.h
SIGNATURES = {
    "msc_selective_scan_fwd_workspace_size": (_sz, [_i64] * 4),
    "msc_selective_scan_fwd": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 11 + [_vp, _sz, _vp]),
    "msc_selective_scan_bwd_workspace_size": (_sz, [_i64] * 4),
    "msc_selective_scan_bwd": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 9 + [_vp] * 8 + [_vp, _sz, _vp]),
    "msc_selective_scan_ckpt_size": (_sz, [_i64] * 4),
    "msc_selective_scan_fwd_train": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 8 + [_vp, _vp] +
                                     [_vp, _sz, _vp]),
    "msc_selective_scan_bwd_ckpt": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 9 + [_vp] + [_vp] * 8 +
                                    [_vp]),
    "msc_ssd_chunked_fwd_workspace_size": (_sz, [_i64] * 7),
    "msc_ssd_chunked_fwd": (ctypes.c_int, [_i64] * 7 + [ctypes.c_int] + [_vp] * 10 + [_vp, _sz, _vp]),
    "msc_ssd_chunked_bwd_workspace_size": (_sz, [_i64] * 7 + [ctypes.c_int]),
    "msc_ssd_chunked_bwd": (ctypes.c_int, [_i64] * 7 + [ctypes.c_int] + [_vp] * 8 + [_vp] * 9 + [_vp, _sz, _vp]),
    "msc_selective_scan_fwd_ex": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] * 2 + [_vp] * 11 + [_vp, _sz, _vp]),
    "msc_selective_scan_fwd_conv": (ctypes.c_int, [_i64] * 5 + [ctypes.c_int] + [_vp] * 13 + [_vp, _sz, _vp]),
    "msc_selective_scan_fwd_noalloc": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 11 + [_vp]),
    "msc_selective_scan_fwd_host_staging_size": (_sz, [_i64] * 4 + [ctypes.c_int] * 2 + [_i64]),
    "msc_selective_scan_fwd_host": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 9 + [_i64, _vp, _sz, _vp]),
    "msc_selective_state_update": (ctypes.c_int, [_i64] * 3 + [ctypes.c_int] + [_vp] * 10 + [_vp]),
    "msc_causal_conv1d_fwd": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] * 2 + [_vp] * 3 + [ctypes.c_int] + [_vp, _vp]),
    "msc_causal_conv1d_update": (ctypes.c_int, [_i64] * 3 + [ctypes.c_int] * 2 + [_vp] * 3 + [ctypes.c_int] + [_vp] * 3),
    "msc_causal_conv1d_bwd": (ctypes.c_int, [_i64] * 4 + [ctypes.c_int] + [_vp] * 3 + [ctypes.c_int] + [_vp] * 5),
    "msc_check_device_status": (ctypes.c_int, [_vp]),
    "msc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "msc_last_error": (ctypes.c_char_p, []),
    "msc_version": (ctypes.c_int, []),
}


class MscError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (_status_name(status), message))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libmsc.so (built in-tree).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    "libmsc.so not found at %s; build it with "
                    "`python -m selective_state_space_160_b300.build`" % _LIB_PATH)
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _status_name(s):
    try:
        return load_library().msc_status_string(int(s)).decode()
    except Exception:  # library missing while formatting an error
        return "status %d" % int(s)


def msc_status_string(s) -> str:
    return load_library().msc_status_string(int(s)).decode()


def msc_last_error() -> str:
    return load_library().msc_last_error().decode()


def _check(status):
    if status != MSC_OK:
        raise MscError(status, msc_last_error())


# ----------------------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _dev_ptr(t, name, dtype=None, shape=None, optional=False):
    torch = _torch()
    if t is None:
        if optional:
            return None
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (this library has no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


def _in_dtype(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return MSC_BF16
    if t.dtype == torch.float32:
        return MSC_F32
    raise ValueError("streamed inputs must be float32 or bfloat16 (got %s)" % t.dtype)


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _workspace(nbytes, device, workspace=None, align=1024):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small: %d < %d bytes" % (workspace.numel(), nbytes))
        return workspace, workspace.numel() * workspace.element_size()
    # torch's caching allocator returns 512-byte aligned blocks; over-allocate
    # and offset for stricter alignment.
    buf = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % align
    return buf[off:off + nbytes], nbytes


# ----------------------------------------------------------------------------- S6
def msc_selective_scan_fwd_workspace_size(batch, dim, seqlen, dstate) -> int:
    return int(load_library().msc_selective_scan_fwd_workspace_size(batch, dim, seqlen, dstate))


def msc_selective_scan_bwd_workspace_size(batch, dim, seqlen, dstate) -> int:
    return int(load_library().msc_selective_scan_bwd_workspace_size(batch, dim, seqlen, dstate))


def msc_selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None,
                           return_last_state=False, y=None, workspace=None, stream=None, disc=MSC_DISC_EULER):
    """S6 forward.  u, delta, z: [batch, dim, L] (fp32 or bf16, all the same);
    B, C: [batch, N, L] (same dtype); A: [dim, N] fp32; D, delta_bias: [dim] fp32;
    h0: [batch, dim, N] fp32.  Returns y [batch, dim, L] fp32 (and h_last).
    disc: MSC_DISC_EULER (msc_selective_scan_fwd), MSC_DISC_ZOH or
    MSC_DISC_TRAPEZOID (msc_selective_scan_fwd_ex)."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    args = [
        _dev_ptr(u, "u"), _dev_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", torch.float32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N, L)), _dev_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", torch.float32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", torch.float32, (dim,), optional=True),
        _dev_ptr(h0, "h0", torch.float32, (batch, dim, N), optional=True),
    ]
    if y is None:
        y = torch.empty((batch, dim, L), dtype=torch.float32, device=u.device)
    h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device) if return_last_state else None
    nbytes = msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    ws, wsb = _workspace(nbytes, u.device, workspace)
    tail = (_dev_ptr(y, "y", torch.float32, (batch, dim, L)), _dev_ptr(h_last, "h_last", optional=True),
            ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    if disc == MSC_DISC_EULER:
        st = lib.msc_selective_scan_fwd(batch, dim, L, N, dt, *args, *tail)
    else:
        st = lib.msc_selective_scan_fwd_ex(batch, dim, L, N, dt, int(disc), *args, *tail)
    _check(st)
    return (y, h_last) if return_last_state else y


def _host_ptr(t, name, dtype=None, shape=None, optional=False):
    torch = _torch()
    if t is None:
        if optional:
            return None
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


def msc_selective_scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, y=None, chunk_batch=1,
                                staging=None, stream=None):
    """S6 forward from and to host memory.  u, delta, z [batch, dim, L] and
    B, C [batch, N, L] are CPU tensors (pinned for overlap), A [dim, N], D and
    delta_bias [dim] CUDA fp32 tensors.  y: CPU fp32 [batch, dim, L] (made
    pinned when None).  The copies of chunk_batch batch entries at a time
    overlap the scan.  Returns y, which is complete once the stream has been
    synchronised (the call itself does not wait)."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    device = A.device
    if y is None:
        y = torch.empty((batch, dim, L), dtype=torch.float32).pin_memory()
    args = [
        _host_ptr(u, "u"), _host_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", torch.float32, (dim, N)),
        _host_ptr(B, "B", tdt, (batch, N, L)), _host_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", torch.float32, (dim,), optional=True),
        _host_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", torch.float32, (dim,), optional=True),
        _host_ptr(y, "y", torch.float32, (batch, dim, L)),
    ]
    nbytes = lib.msc_selective_scan_fwd_host_staging_size(batch, dim, L, N, dt, int(z is not None), chunk_batch)
    ws, wsb = _workspace(nbytes, device, staging, align=256)
    _check(lib.msc_selective_scan_fwd_host(batch, dim, L, N, dt, *args, chunk_batch,
                                           ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream)))
    return y


def msc_selective_scan_fwd_conv(x, conv_weight, conv_bias, delta, A, B, C, D=None, z=None, delta_bias=None,
                                h0=None, return_last_state=False, y=None, workspace=None, stream=None):
    """S6 forward with the causal conv1d + SiLU front end fused: u =
    silu(conv_bias + causal depthwise conv of x with conv_weight [dim, width])
    is formed inside the scan.  x, delta, z: [batch, dim, L] (fp32 or bf16, all
    the same); conv_weight [dim, width <= 4] fp32; conv_bias [dim] fp32 or None;
    the rest as msc_selective_scan_fwd.  Returns y (and h_last)."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = x.shape
    N = A.shape[1]
    K = conv_weight.shape[1]
    dt = _in_dtype(x)
    tdt = x.dtype
    if y is None:
        y = torch.empty((batch, dim, L), dtype=torch.float32, device=x.device)
    h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=x.device) if return_last_state else None
    nbytes = msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    ws, wsb = _workspace(nbytes, x.device, workspace)
    st = lib.msc_selective_scan_fwd_conv(
        batch, dim, L, N, K, dt, _dev_ptr(x, "x"),
        _dev_ptr(conv_weight, "conv_weight", torch.float32, (dim, K)),
        _dev_ptr(conv_bias, "conv_bias", torch.float32, (dim,), optional=True),
        _dev_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", torch.float32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N, L)), _dev_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", torch.float32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", torch.float32, (dim,), optional=True),
        _dev_ptr(h0, "h0", torch.float32, (batch, dim, N), optional=True),
        _dev_ptr(y, "y", torch.float32, (batch, dim, L)), _dev_ptr(h_last, "h_last", optional=True),
        ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    _check(st)
    return (y, h_last) if return_last_state else y


def msc_selective_state_update(u, delta, A, B, C, D=None, z=None, delta_bias=None, state=None,
                               y=None, stream=None):
    """S6 decode step: one token per row.  u, delta, z: [batch, dim] (fp32 or
    bf16, all the same); B, C: [batch, N] (same dtype); A: [dim, N] fp32;
    D, delta_bias: [dim] fp32; state: [batch, dim, N] fp32, updated in place.
    Returns y [batch, dim] fp32."""
    torch = _torch()
    lib = load_library()
    if state is None:
        raise ValueError("state is required (it is read and updated in place)")
    batch, dim = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    args = [
        _dev_ptr(u, "u"), _dev_ptr(delta, "delta", tdt, (batch, dim)),
        _dev_ptr(A, "A", torch.float32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N)), _dev_ptr(C, "C", tdt, (batch, N)),
        _dev_ptr(D, "D", torch.float32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim), optional=True),
        _dev_ptr(delta_bias, "delta_bias", torch.float32, (dim,), optional=True),
        _dev_ptr(state, "state", torch.float32, (batch, dim, N)),
    ]
    if y is None:
        y = torch.empty((batch, dim), dtype=torch.float32, device=u.device)
    st = lib.msc_selective_state_update(batch, dim, N, dt, *args, _dev_ptr(y, "y", torch.float32, (batch, dim)),
                                        _stream_ptr(stream))
    _check(st)
    return y


def _dtype_code(dtype):
    torch = _torch()
    if dtype == torch.float32:
        return MSC_F32
    if dtype == torch.bfloat16:
        return MSC_BF16
    raise ValueError("dtype must be torch.float32 or torch.bfloat16 (got %s)" % dtype)


def msc_causal_conv1d_fwd(x, weight, bias=None, silu=True, out_dtype=None, out=None, stream=None):
    """Causal depthwise conv1d (+ SiLU).  x: [batch, dim, L] fp32 or bf16;
    weight: [dim, K] fp32; bias: [dim] fp32.  Returns out [batch, dim, L] in
    out_dtype (default: x's dtype), ready to be the scan's u."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = x.shape
    K = weight.shape[1]
    out_dtype = x.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((batch, dim, L), dtype=out_dtype, device=x.device)
    st = lib.msc_causal_conv1d_fwd(batch, dim, L, K, _in_dtype(x), _dtype_code(out.dtype), _dev_ptr(x, "x"),
                                   _dev_ptr(weight, "weight", torch.float32, (dim, K)),
                                   _dev_ptr(bias, "bias", torch.float32, (dim,), optional=True), int(bool(silu)),
                                   _dev_ptr(out, "out", out.dtype, (batch, dim, L)), _stream_ptr(stream))
    _check(st)
    return out


def msc_causal_conv1d_bwd(x, weight, dout, bias=None, silu=True, with_dbias=True, stream=None):
    """Backward of msc_causal_conv1d_fwd.  x: [batch, dim, L] fp32 or bf16;
    weight [dim, K], bias [dim] fp32 (the forward's); dout [batch, dim, L] fp32.
    Returns (dx [batch, dim, L], dweight [dim, K], dbias [dim] or None), fp32."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = x.shape
    K = weight.shape[1]
    f32 = torch.float32
    dx = torch.empty((batch, dim, L), dtype=f32, device=x.device)
    dw = torch.empty((dim, K), dtype=f32, device=x.device)
    db = torch.empty((dim,), dtype=f32, device=x.device) if with_dbias else None
    st = lib.msc_causal_conv1d_bwd(batch, dim, L, K, _in_dtype(x), _dev_ptr(x, "x"),
                                   _dev_ptr(weight, "weight", f32, (dim, K)),
                                   _dev_ptr(bias, "bias", f32, (dim,), optional=True), int(bool(silu)),
                                   _dev_ptr(dout, "dout", f32, (batch, dim, L)), _dev_ptr(dx, "dx"),
                                   _dev_ptr(dw, "dweight"), _dev_ptr(db, "dbias", optional=True), _stream_ptr(stream))
    _check(st)
    return dx, dw, db


def msc_causal_conv1d_update(x, conv_state, weight, bias=None, silu=True, out_dtype=None, out=None, stream=None):
    """Decode step of the causal conv1d.  x: [batch, dim]; conv_state:
    [batch, dim, K - 1] fp32, updated in place.  Returns out [batch, dim]."""
    torch = _torch()
    lib = load_library()
    batch, dim = x.shape
    K = weight.shape[1]
    out_dtype = x.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((batch, dim), dtype=out_dtype, device=x.device)
    state_ptr = _dev_ptr(conv_state, "conv_state", torch.float32, (batch, dim, K - 1), optional=(K == 1))
    st = lib.msc_causal_conv1d_update(batch, dim, K, _in_dtype(x), _dtype_code(out.dtype), _dev_ptr(x, "x"),
                                      _dev_ptr(weight, "weight", torch.float32, (dim, K)),
                                      _dev_ptr(bias, "bias", torch.float32, (dim,), optional=True),
                                      int(bool(silu)), state_ptr, _dev_ptr(out, "out", out.dtype, (batch, dim)),
                                      _stream_ptr(stream))
    _check(st)
    return out


def msc_selective_scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, dy=None,
                           workspace=None, stream=None):
    """S6 backward (zero initial state).  Returns a dict with du, ddelta, dA, dB,
    dC and, when the matching input is given, dD, dz, ddelta_bias (all fp32)."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    dev = u.device
    f32 = torch.float32
    out = {
        "du": torch.empty((batch, dim, L), dtype=f32, device=dev),
        "ddelta": torch.empty((batch, dim, L), dtype=f32, device=dev),
        "dA": torch.empty((dim, N), dtype=f32, device=dev),
        "dB": torch.empty((batch, N, L), dtype=f32, device=dev),
        "dC": torch.empty((batch, N, L), dtype=f32, device=dev),
        "dD": torch.empty((dim,), dtype=f32, device=dev) if D is not None else None,
        "dz": torch.empty((batch, dim, L), dtype=f32, device=dev) if z is not None else None,
        "ddelta_bias": torch.empty((dim,), dtype=f32, device=dev) if delta_bias is not None else None,
    }
    nbytes = msc_selective_scan_bwd_workspace_size(batch, dim, L, N)
    ws, wsb = _workspace(nbytes, dev, workspace)
    st = lib.msc_selective_scan_bwd(
        batch, dim, L, N, dt,
        _dev_ptr(u, "u"), _dev_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", f32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N, L)), _dev_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", f32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", f32, (dim,), optional=True),
        _dev_ptr(dy, "dy", tdt, (batch, dim, L)),
        *[(_dev_ptr(out[k], k, optional=True)) for k in
          ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")],
        ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    _check(st)
    return out


def msc_selective_scan_ckpt_size(batch, dim, seqlen, dstate) -> int:
    return int(load_library().msc_selective_scan_ckpt_size(batch, dim, seqlen, dstate))


def msc_selective_scan_fwd_train(u, delta, A, B, C, D=None, z=None, delta_bias=None, y=None, ckpt=None,
                                 workspace=None, stream=None):
    """Training forward: y as msc_selective_scan_fwd (zero initial state) and the
    backward's checkpoints (fp32, [batch * dim, L / 8, 16]).  Returns (y, ckpt)."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    f32 = torch.float32
    if y is None:
        y = torch.empty((batch, dim, L), dtype=f32, device=u.device)
    if ckpt is None:
        ckpt = torch.empty((batch * dim, max(L // 8, 1), 16), dtype=f32, device=u.device)
    nbytes = msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    ws, wsb = _workspace(nbytes, u.device, workspace)
    st = lib.msc_selective_scan_fwd_train(
        batch, dim, L, N, dt,
        _dev_ptr(u, "u"), _dev_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", f32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N, L)), _dev_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", f32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", f32, (dim,), optional=True),
        _dev_ptr(y, "y", f32, (batch, dim, L)), _dev_ptr(ckpt, "ckpt", f32),
        ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    _check(st)
    return y, ckpt


def msc_selective_scan_bwd_ckpt(u, delta, A, B, C, D=None, z=None, delta_bias=None, dy=None, ckpt=None,
                                stream=None):
    """S6 backward from the training forward's checkpoints; gradients as
    msc_selective_scan_bwd (a dict), no workspace."""
    torch = _torch()
    lib = load_library()
    batch, dim, L = u.shape
    N = A.shape[1]
    dt = _in_dtype(u)
    tdt = u.dtype
    dev = u.device
    f32 = torch.float32
    out = {
        "du": torch.empty((batch, dim, L), dtype=f32, device=dev),
        "ddelta": torch.empty((batch, dim, L), dtype=f32, device=dev),
        "dA": torch.empty((dim, N), dtype=f32, device=dev),
        "dB": torch.empty((batch, N, L), dtype=f32, device=dev),
        "dC": torch.empty((batch, N, L), dtype=f32, device=dev),
        "dD": torch.empty((dim,), dtype=f32, device=dev) if D is not None else None,
        "dz": torch.empty((batch, dim, L), dtype=f32, device=dev) if z is not None else None,
        "ddelta_bias": torch.empty((dim,), dtype=f32, device=dev) if delta_bias is not None else None,
    }
    st = lib.msc_selective_scan_bwd_ckpt(
        batch, dim, L, N, dt,
        _dev_ptr(u, "u"), _dev_ptr(delta, "delta", tdt, (batch, dim, L)),
        _dev_ptr(A, "A", f32, (dim, N)),
        _dev_ptr(B, "B", tdt, (batch, N, L)), _dev_ptr(C, "C", tdt, (batch, N, L)),
        _dev_ptr(D, "D", f32, (dim,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, dim, L), optional=True),
        _dev_ptr(delta_bias, "delta_bias", f32, (dim,), optional=True),
        _dev_ptr(dy, "dy", tdt, (batch, dim, L)), _dev_ptr(ckpt, "ckpt", f32),
        *[(_dev_ptr(out[k], k, optional=True)) for k in
          ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")],
        _stream_ptr(stream))
    _check(st)
    return out


# ----------------------------------------------------------------------------- SSD
def msc_ssd_chunked_fwd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, chunk) -> int:
    return int(load_library().msc_ssd_chunked_fwd_workspace_size(batch, seqlen, nheads, headdim,
                                                                 dstate, ngroups, chunk))


def msc_ssd_chunked_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, chunk=256,
                        return_final_state=False, y=None, workspace=None, stream=None,
                        return_workspace=False):
    """SSD forward.  x, z: [batch, L, heads, P] bf16; delta: [batch, L, heads] bf16;
    A, D, delta_bias: [heads] fp32; B, C: [batch, L, groups, N] bf16.
    Returns y [batch, L, heads, P] fp32 (and the final state [batch, heads, P, N])."""
    torch = _torch()
    lib = load_library()
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dt = _in_dtype(x)
    tdt = x.dtype
    f32 = torch.float32
    dev = x.device
    if y is None:
        y = torch.empty((batch, L, H, P), dtype=f32, device=dev)
    fs = torch.empty((batch, H, P, N), dtype=f32, device=dev) if return_final_state else None
    nbytes = msc_ssd_chunked_fwd_workspace_size(batch, L, H, P, N, G, chunk)
    ws, wsb = _workspace(nbytes, dev, workspace)
    st = lib.msc_ssd_chunked_fwd(
        batch, L, H, P, N, G, chunk, dt,
        _dev_ptr(x, "x"), _dev_ptr(delta, "delta", tdt, (batch, L, H)),
        _dev_ptr(A, "A", f32, (H,)),
        _dev_ptr(B, "B", tdt, (batch, L, G, N)), _dev_ptr(C, "C", tdt, (batch, L, G, N)),
        _dev_ptr(D, "D", f32, (H,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, L, H, P), optional=True),
        _dev_ptr(delta_bias, "delta_bias", f32, (H,), optional=True),
        _dev_ptr(y, "y", f32, (batch, L, H, P)), _dev_ptr(fs, "final_state", optional=True),
        ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    _check(st)
    res = (y, fs) if return_final_state else y
    if return_workspace:
        return res, ws
    return res


def msc_ssd_chunked_bwd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, chunk,
                                       has_z) -> int:
    return int(load_library().msc_ssd_chunked_bwd_workspace_size(batch, seqlen, nheads, headdim,
                                                                 dstate, ngroups, chunk, int(bool(has_z))))


def msc_ssd_chunked_bwd(x, delta, A, B, C, dy, D=None, z=None, delta_bias=None, chunk=256,
                        workspace=None, stream=None):
    """SSD backward (zero initial state).  Inputs as msc_ssd_chunked_fwd plus
    dy [batch, L, heads, P] bf16.  Returns a dict of fp32 gradients dx, ddelta,
    dA, dB, dC and, for the optional inputs given, dD, dz, ddelta_bias."""
    torch = _torch()
    lib = load_library()
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dt = _in_dtype(x)
    tdt = x.dtype
    f32 = torch.float32
    dev = x.device
    g = {"dx": torch.empty((batch, L, H, P), dtype=f32, device=dev),
         "ddelta": torch.empty((batch, L, H), dtype=f32, device=dev),
         "dA": torch.empty((H,), dtype=f32, device=dev),
         "dB": torch.empty((batch, L, G, N), dtype=f32, device=dev),
         "dC": torch.empty((batch, L, G, N), dtype=f32, device=dev),
         "dD": torch.empty((H,), dtype=f32, device=dev) if D is not None else None,
         "dz": torch.empty((batch, L, H, P), dtype=f32, device=dev) if z is not None else None,
         "ddelta_bias": torch.empty((H,), dtype=f32, device=dev) if delta_bias is not None else None}
    nbytes = msc_ssd_chunked_bwd_workspace_size(batch, L, H, P, N, G, chunk, z is not None)
    ws, wsb = _workspace(nbytes, dev, workspace)
    st = lib.msc_ssd_chunked_bwd(
        batch, L, H, P, N, G, chunk, dt,
        _dev_ptr(x, "x"), _dev_ptr(delta, "delta", tdt, (batch, L, H)),
        _dev_ptr(A, "A", f32, (H,)),
        _dev_ptr(B, "B", tdt, (batch, L, G, N)), _dev_ptr(C, "C", tdt, (batch, L, G, N)),
        _dev_ptr(D, "D", f32, (H,), optional=True),
        _dev_ptr(z, "z", tdt, (batch, L, H, P), optional=True),
        _dev_ptr(delta_bias, "delta_bias", f32, (H,), optional=True),
        _dev_ptr(dy, "dy", tdt, (batch, L, H, P)),
        _dev_ptr(g["dx"], "dx"), _dev_ptr(g["ddelta"], "ddelta"), _dev_ptr(g["dA"], "dA"),
        _dev_ptr(g["dB"], "dB"), _dev_ptr(g["dC"], "dC"),
        _dev_ptr(g["dD"], "dD", optional=True), _dev_ptr(g["dz"], "dz", optional=True),
        _dev_ptr(g["ddelta_bias"], "ddelta_bias", optional=True),
        ws.data_ptr() if ws is not None else None, wsb, _stream_ptr(stream))
    _check(st)
    return {k: v for k, v in g.items() if v is not None}


def msc_check_device_status(stream=None):
    """Synchronise the stream and raise if device code recorded an error
    (a bounded wait that ran out); reading clears the recorded error."""
    _check(load_library().msc_check_device_status(_stream_ptr(stream)))
