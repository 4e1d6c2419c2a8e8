"""ctypes wrapper around the double-precision CPU oracle (msc_oracle.c).

TEST INFRASTRUCTURE.  Only tests/, ``__graft_entry__.smoke()`` and bench.py's
CPU-baseline leg may import this module.  It shares nothing with the CUDA library
and never touches the GPU.  Inputs are converted to float64 exactly (fp32 and
bf16-rounded values are exact in double), outputs are float64.

The S6 forward, its backward, the decode step and the SSD forward are computed
in msc_oracle.c (plain C, double); this file marshals their arrays.  Four
oracle functions are written here in numpy, in float64: the causal conv1d with
SiLU, its decode step and its backward, and the SSD backward (the S6 backward
composed over the channels that share a head's Delta and A and a group's B, C).
Parity of each function is pinned in tests/test_oracle_pins.py (closed forms, special
cases, brute force and finite differences), so none of them is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msc_oracle.c")
_LIB = os.path.join(_HERE, "libmsc_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile msc_oracle.c with gcc (-O2, no fast-math, OpenMP) in place."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_s6_fwd.argtypes = [_i64] * 4 + [_dp] * 11
            lib.oracle_s6_fwd.restype = ctypes.c_int
            lib.oracle_s6_bwd.argtypes = [_i64] * 4 + [_dp] * 17
            lib.oracle_s6_bwd.restype = ctypes.c_int
            lib.oracle_s6_fwd_disc.argtypes = [ctypes.c_int] + [_i64] * 4 + [_dp] * 11
            lib.oracle_s6_fwd_disc.restype = ctypes.c_int
            lib.oracle_ssd_fwd.argtypes = [_i64] * 6 + [_dp] * 10
            lib.oracle_ssd_fwd.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.cast(None, _dp)
    return a.ctypes.data_as(_dp)


def s6_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None,
           return_last_state=False):
    """S6 forward.  u, delta, z: [batch, dim, L]; A: [dim, N]; B, C: [batch, N, L];
    D, delta_bias: [dim]; h0: [batch, dim, N].  Returns y (and h_last)."""
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, z, delta_bias, h0 = map(_f64, (D, z, delta_bias, h0))
    batch, dim, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and A.shape == (dim, N)
    assert B.shape == (batch, N, L) and C.shape == (batch, N, L)
    y = np.empty((batch, dim, L), np.float64)
    h_last = np.empty((batch, dim, N), np.float64)
    rc = _load().oracle_s6_fwd(batch, dim, L, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                               _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0),
                               _ptr(y), _ptr(h_last))
    if rc:
        raise MemoryError("oracle_s6_fwd failed")
    return (y, h_last) if return_last_state else y


DISC_EULER, DISC_ZOH, DISC_TRAPEZOID = 0, 1, 2


def s6_fwd_disc(disc, u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None,
                return_last_state=False):
    """S6 forward with the input term discretised by zero-order hold (disc 1,
    "Mamba 解密" sec. 3 / sec. 5) or by the exponential-trapezoidal rule (disc 2,
    "Mamba 解密" sec. 6.3); disc 0 is the exponential-Euler s6_fwd.  Same
    shapes and results as s6_fwd."""
    if disc == DISC_EULER:
        return s6_fwd(u, delta, A, B, C, D, z, delta_bias, h0, return_last_state)
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, z, delta_bias, h0 = map(_f64, (D, z, delta_bias, h0))
    batch, dim, L = u.shape
    N = A.shape[1]
    assert delta.shape == u.shape and A.shape == (dim, N)
    assert B.shape == (batch, N, L) and C.shape == (batch, N, L)
    y = np.empty((batch, dim, L), np.float64)
    h_last = np.empty((batch, dim, N), np.float64)
    rc = _load().oracle_s6_fwd_disc(int(disc), batch, dim, L, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                                    _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(y),
                                    _ptr(h_last))
    if rc:
        raise ValueError("oracle_s6_fwd_disc failed (%d)" % rc)
    return (y, h_last) if return_last_state else y


def s6_step(u, delta, A, B, C, D=None, z=None, delta_bias=None, state=None):
    """One decode step ("Mamba — 选择性状态空间模型", 实践案例 1: one token updates the
    fixed-size state once and is read out): the forward recurrence over a
    single step from `state`.  u, delta, z: [batch, dim]; B, C: [batch, N];
    state: [batch, dim, N] (zero if None).  Returns (y [batch, dim], new state)."""
    u, delta, B, C = map(_f64, (u, delta, B, C))
    z = None if z is None else _f64(z)[:, :, None]
    y, h = s6_fwd(u[:, :, None], delta[:, :, None], A, B[:, :, None], C[:, :, None], D, z, delta_bias,
                  state, return_last_state=True)
    return y[:, :, 0], h


def _silu(v):
    return v / (1.0 + np.exp(-v))


def causal_conv1d(x, weight, bias=None, silu=True):
    """Causal depthwise conv1d front end of the Mamba block (bqwf survey sec. 3.1:
    a causal 1-D convolution for local context before the selective SSM):
    out[b, d, t] = act(bias[d] + sum_k weight[d, k] x[b, d, t - (K - 1) + k]),
    x = 0 before t = 0, act = silu or identity.  x: [batch, dim, L];
    weight: [dim, K]; bias: [dim]."""
    x = _f64(x)
    w = _f64(weight)
    batch, dim, L = x.shape
    K = w.shape[1]
    xp = np.concatenate([np.zeros((batch, dim, K - 1)), x], axis=2)
    out = np.zeros((batch, dim, L)) if bias is None else np.broadcast_to(_f64(bias)[None, :, None],
                                                                          (batch, dim, L)).copy()
    for k in range(K):
        out += w[None, :, k, None] * xp[:, :, k:k + L]
    return _silu(out) if silu else out


def causal_conv1d_update(x, conv_state, weight, bias=None, silu=True):
    """Decode step of causal_conv1d (study note "Mamba — 选择性状态空间模型",
    踩过的坑: the convolution keeps the last few inputs).  x: [batch, dim];
    conv_state: [batch, dim, K - 1], oldest first.  Returns (out, new state)."""
    x = _f64(x)
    w = _f64(weight)
    window = np.concatenate([_f64(conv_state), x[:, :, None]], axis=2)
    out = np.einsum("bdk,dk->bd", window, w)
    if bias is not None:
        out = out + _f64(bias)[None, :]
    return (_silu(out) if silu else out), window[:, :, 1:]


def causal_conv1d_bwd(x, weight, bias=None, dout=None, silu=True):
    """Gradients of causal_conv1d for an upstream gradient dout [batch, dim, L]
    (the chain rule through its definition): with pre the pre-activation and
    g = dout * silu'(pre) (g = dout without the activation),
      dx[b, d, s]  = sum_k weight[d, k] g[b, d, s + (K - 1) - k]   (terms past L are 0)
      dweight[d, k] = sum_{b, t} g[b, d, t] x[b, d, t - (K - 1) + k]
      dbias[d]     = sum_{b, t} g[b, d, t].
    Returns (dx, dweight, dbias) in float64."""
    x = _f64(x)
    w = _f64(weight)
    g = _f64(dout)
    batch, dim, L = x.shape
    K = w.shape[1]
    if silu:
        pre = causal_conv1d(x, w, bias, silu=False)
        sg = 1.0 / (1.0 + np.exp(-pre))
        g = g * sg * (1.0 + pre * (1.0 - sg))
    xp = np.concatenate([np.zeros((batch, dim, K - 1)), x], axis=2)
    gp = np.concatenate([g, np.zeros((batch, dim, K - 1))], axis=2)
    dx = np.zeros((batch, dim, L))
    dw = np.zeros((dim, K))
    for k in range(K):
        dx += w[None, :, k, None] * gp[:, :, K - 1 - k:K - 1 - k + L]
        dw[:, k] = np.einsum("bdt,bdt->d", g, xp[:, :, k:k + L])
    return dx, dw, g.sum(axis=(0, 2))


def s6_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, dy=None):
    """S6 backward (zero initial state).  Returns a dict of float64 grads:
    du, ddelta, dA, dB, dC, and dD / dz / ddelta_bias when the input is present."""
    u, delta, A, B, C, dy = map(_f64, (u, delta, A, B, C, dy))
    D, z, delta_bias = map(_f64, (D, z, delta_bias))
    batch, dim, L = u.shape
    N = A.shape[1]
    out = {
        "du": np.empty_like(u), "ddelta": np.empty_like(u),
        "dA": np.empty((dim, N)), "dB": np.empty((batch, N, L)), "dC": np.empty((batch, N, L)),
        "dD": np.empty(dim), "dz": np.empty_like(u) if z is not None else None,
        "ddelta_bias": np.empty(dim),
    }
    rc = _load().oracle_s6_bwd(batch, dim, L, N, _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                               _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(dy),
                               _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]),
                               _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                               _ptr(out["dz"]), _ptr(out["ddelta_bias"]))
    if rc:
        raise MemoryError("oracle_s6_bwd failed")
    if D is None:
        out["dD"] = None
    if delta_bias is None:
        out["ddelta_bias"] = None
    return out


def ssd_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, return_final_state=False):
    """SSD forward.  x, z: [batch, L, heads, P]; delta: [batch, L, heads];
    A, D, delta_bias: [heads]; B, C: [batch, L, groups, N]."""
    x, delta, A, B, C = map(_f64, (x, delta, A, B, C))
    D, z, delta_bias = map(_f64, (D, z, delta_bias))
    batch, L, nheads, P = x.shape
    ngroups, N = B.shape[2], B.shape[3]
    y = np.empty_like(x)
    fs = np.empty((batch, nheads, P, N))
    rc = _load().oracle_ssd_fwd(batch, L, nheads, P, N, ngroups, _ptr(x), _ptr(delta),
                                _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                _ptr(delta_bias), _ptr(y), _ptr(fs))
    if rc:
        raise ValueError("oracle_ssd_fwd failed (rc=%d)" % rc)
    return (y, fs) if return_final_state else y


def ssd_bwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, dy=None):
    """SSD backward (zero initial state).  The SSD is the S6 scan with channels
    d = (head, p), Delta and A shared by a head's P channels and B, C shared by
    a group's heads (bqwf survey sec. 3.2: scalar A_t = alpha_t I); so each
    gradient is the S6 backward of that problem, summed over the channels that
    share the parameter: dx = du; ddelta[h] = sum_p ddelta(h, p); dA[h] =
    sum_{p,n} dA(h, p, n); dD, ddelta_bias likewise; dB, dC per group.
    Shapes as ssd_fwd; returns a dict dx, ddelta, dA, dB, dC and, when the input
    is given, dD, dz, ddelta_bias."""
    x, delta, A, B, C, dy = map(_f64, (x, delta, A, B, C, dy))
    D, z, delta_bias = map(_f64, (D, z, delta_bias))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    out = {"dx": np.empty_like(x), "ddelta": np.empty((batch, L, H)), "dA": np.empty(H),
           "dB": np.empty_like(B), "dC": np.empty_like(C),
           "dD": np.empty(H) if D is not None else None, "dz": np.empty_like(x) if z is not None else None,
           "ddelta_bias": np.empty(H) if delta_bias is not None else None}
    for g in range(G):
        heads = list(range(g * hpg, (g + 1) * hpg))
        u = np.concatenate([x[:, :, h, :].transpose(0, 2, 1) for h in heads], axis=1)
        dl = np.concatenate([np.repeat(delta[:, None, :, h], P, axis=1) for h in heads], axis=1)
        dyy = np.concatenate([dy[:, :, h, :].transpose(0, 2, 1) for h in heads], axis=1)
        zz = None if z is None else np.concatenate([z[:, :, h, :].transpose(0, 2, 1) for h in heads], axis=1)
        A6 = np.concatenate([np.full((P, N), A[h]) for h in heads], axis=0)
        D6 = None if D is None else np.concatenate([np.full(P, D[h]) for h in heads])
        b6 = None if delta_bias is None else np.concatenate([np.full(P, delta_bias[h]) for h in heads])
        r = s6_bwd(u, dl, A6, B[:, :, g, :].transpose(0, 2, 1), C[:, :, g, :].transpose(0, 2, 1), D6, zz, b6, dyy)
        out["dB"][:, :, g, :] = r["dB"].transpose(0, 2, 1)
        out["dC"][:, :, g, :] = r["dC"].transpose(0, 2, 1)
        for i, h in enumerate(heads):
            sl = slice(i * P, (i + 1) * P)
            out["dx"][:, :, h, :] = r["du"][:, sl, :].transpose(0, 2, 1)
            out["ddelta"][:, :, h] = r["ddelta"][:, sl, :].sum(axis=1)
            out["dA"][h] = r["dA"][sl].sum()
            if D is not None:
                out["dD"][h] = r["dD"][sl].sum()
            if z is not None:
                out["dz"][:, :, h, :] = r["dz"][:, sl, :].transpose(0, 2, 1)
            if delta_bias is not None:
                out["ddelta_bias"][h] = r["ddelta_bias"][sl].sum()
    return out
