"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own loop.  Each compares it with an
independent statement of the same quantity:

  P1 materialised closed form of the S6 output (sum over sources s <= t of the
     explicit decay products), written with numpy on tiny inputs;
  P2 Delta -> 0 leaves only the feed-through D * u (times the gate);
  P3 constant Delta, B, C: the scan is an LTI causal convolution (numpy.convolve
     and an FFT convolution);
  P4 SSD: the materialised semiseparable form y_i = sum_{j<=i} M_ij (C_i.B_j) Delta_j x_j
     with M_ij = a_{j+1}...a_i, the S6 oracle with channels (head, p), and a
     chunked block decomposition all agree;
  P5 central finite differences of <w, y> against the hand-derived backward;
  P6 linearity in u and the split scan [0,L) = [0,k) then [k,L) from h_last;
  P7 the decay bound |h_t| <= sum |Delta B u| when A < 0;
  P8 a single step and the study note's worked three-step recurrence by hand.
A planted mistake in the oracle (a dropped term, a wrong sign or index, a
transposed operand) fails at least one of them; test_planted_mistakes checks
that on CPU copies of the oracle with such mistakes.
"""
import os
import shutil
import subprocess
import ctypes

import numpy as np
import pytest
from scipy.special import expit
from scipy.signal import fftconvolve

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, ssd_inputs


def softplus(x):
    return np.logaddexp(0.0, x)


def silu(z):
    return z * expit(z)


def closed_form_s6(u, delta, A, B, C, D=None, z=None, bias=None):
    """P1: y_t = [sum_{s<=t} sum_n C_tn (prod_{r=s+1..t} exp(Delta_r A_n)) Delta_s B_sn u_s
    + D u_t] * silu(z_t), by explicit products (O(L^2 N))."""
    f64 = lambda a: None if a is None else np.asarray(a, np.float64)
    u, delta, A, B, C, D, z, bias = map(f64, (u, delta, A, B, C, D, z, bias))
    batch, dim, L = u.shape
    N = A.shape[1]
    y = np.zeros((batch, dim, L))
    for b in range(batch):
        for d in range(dim):
            dt = softplus(delta[b, d].astype(np.float64) + (bias[d] if bias is not None else 0.0))
            for t in range(L):
                acc = 0.0
                for s in range(t + 1):
                    decay = np.ones(N)
                    for r in range(s + 1, t + 1):
                        decay = decay * np.exp(dt[r] * A[d])
                    acc += np.sum(C[b, :, t] * decay * dt[s] * B[b, :, s] * u[b, d, s])
                if D is not None:
                    acc += D[d] * u[b, d, t]
                if z is not None:
                    acc *= silu(z[b, d, t])
                y[b, d, t] = acc
    return y


def rel_err(a, b):
    return float(np.max(np.abs(a - b) / (1.0 + np.abs(b))))


@pytest.fixture(scope="module")
def tiny():
    return s6_inputs(2, 4, 24, 5, seed=11)


# ----------------------------------------------------------------------------- P1
@pytest.mark.parametrize("with_z,with_D,with_bias", [(True, True, True), (False, True, True),
                                                     (True, False, False), (False, False, True)])
def test_p1_closed_form(with_z, with_D, with_bias):
    inp = s6_inputs(1, 3, 20, 4, seed=3, with_z=with_z, with_D=with_D, with_bias=with_bias)
    y = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                      inp["z"], inp["delta_bias"])
    ref = closed_form_s6(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                         inp["z"], inp["delta_bias"])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_p1_closed_form_config0_shape():
    # tiny fp32 configuration: batch 1, 4 channels, L = 64, N = 16
    inp = s6_inputs(1, 4, 64, 16, seed=160_000)
    y = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                      inp["z"], inp["delta_bias"])
    ref = closed_form_s6(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                         inp["z"], inp["delta_bias"])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- P2
def test_p2_zero_delta_feedthrough(tiny):
    inp = {k: (None if v is None else np.asarray(v, np.float64)) for k, v in tiny.items()}
    bias = np.full(inp["A"].shape[0], -200.0)   # softplus(-200) ~ 1e-87 -> Delta = 0
    y = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                      inp["z"], bias)
    ref = inp["D"][None, :, None] * inp["u"] * silu(inp["z"].astype(np.float64))
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- P3
def test_p3_lti_convolution():
    rng = np.random.default_rng(5)
    batch, dim, L, N = 1, 3, 96, 6
    u = rng.standard_normal((batch, dim, L))
    delta = np.repeat(rng.standard_normal((batch, dim, 1)) * 0.5, L, axis=2)
    A = -rng.uniform(0.1, 3.0, size=(dim, N))
    Bc = rng.standard_normal((batch, N, 1))
    Cc = rng.standard_normal((batch, N, 1))
    B = np.repeat(Bc, L, axis=2)
    C = np.repeat(Cc, L, axis=2)
    D = rng.standard_normal(dim)
    bias = rng.standard_normal(dim) * 0.3
    y = oracle.s6_fwd(u, delta, A, B, C, D, None, bias)
    k = np.arange(L)
    for d in range(dim):
        dt = softplus(delta[0, d, 0] + bias[d])
        K = np.array([np.sum(Cc[0, :, 0] * np.exp(kk * dt * A[d]) * dt * Bc[0, :, 0]) for kk in k])
        direct = np.convolve(K, u[0, d])[:L] + D[d] * u[0, d]
        viafft = fftconvolve(K, u[0, d])[:L] + D[d] * u[0, d]
        np.testing.assert_allclose(y[0, d], direct, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(y[0, d], viafft, rtol=1e-9, atol=1e-10)


# ----------------------------------------------------------------------------- P4
def materialised_ssd(x, delta, A, B, C, D=None, z=None, bias=None):
    """y_i = sum_{j<=i} M_ij (C_i . B_j) Delta_j x_j + D x_i with M_ij = a_{j+1} ... a_i."""
    f64 = lambda a: None if a is None else np.asarray(a, np.float64)
    x, delta, A, B, C, D, z, bias = map(f64, (x, delta, A, B, C, D, z, bias))
    batch, L, H, P = x.shape
    G = B.shape[2]
    hpg = H // G
    y = np.zeros((batch, L, H, P))
    for b in range(batch):
        for h in range(H):
            g = h // hpg
            dt = softplus(delta[b, :, h].astype(np.float64) + (bias[h] if bias is not None else 0.0))
            a = np.exp(dt * A[h])
            M = np.zeros((L, L))
            for i in range(L):
                for j in range(i + 1):
                    M[i, j] = np.prod(a[j + 1:i + 1])   # empty product = 1 on the diagonal
            CB = C[b, :, g, :].astype(np.float64) @ B[b, :, g, :].astype(np.float64).T
            Y = (M * CB) @ (dt[:, None] * x[b, :, h, :])
            if D is not None:
                Y = Y + D[h] * x[b, :, h, :]
            if z is not None:
                Y = Y * silu(z[b, :, h, :].astype(np.float64))
            y[b, :, h, :] = Y
    return y


def chunked_ssd(x, delta, A, B, C, Q, D=None, bias=None):
    """Block decomposition: intra-chunk masked matmul + inter-chunk state passing."""
    f64 = lambda a: None if a is None else np.asarray(a, np.float64)
    x, delta, A, B, C, D, bias = map(f64, (x, delta, A, B, C, D, bias))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    y = np.zeros((batch, L, H, P))
    for b in range(batch):
        for h in range(H):
            g = h // hpg
            dt = softplus(delta[b, :, h].astype(np.float64) + (bias[h] if bias is not None else 0.0))
            la = dt * A[h]                       # log a_t
            S = np.zeros((P, N))                 # state entering the chunk
            for c0 in range(0, L, Q):
                c1 = min(c0 + Q, L)
                cs = np.cumsum(la[c0:c1])        # inclusive within the chunk
                n = c1 - c0
                Lmat = np.zeros((n, n))
                for i in range(n):
                    for j in range(i + 1):
                        Lmat[i, j] = np.exp(cs[i] - cs[j])
                Cc = C[b, c0:c1, g, :].astype(np.float64)
                Bc = B[b, c0:c1, g, :].astype(np.float64)
                Xd = dt[c0:c1, None] * x[b, c0:c1, h, :]
                Ydiag = (Lmat * (Cc @ Bc.T)) @ Xd
                Yoff = np.exp(cs)[:, None] * (Cc @ S.T)
                Yc = Ydiag + Yoff
                if D is not None:
                    Yc = Yc + D[h] * x[b, c0:c1, h, :]
                y[b, c0:c1, h, :] = Yc
                w = np.exp(cs[-1] - cs)          # decay from step j to the chunk end
                S = np.exp(cs[-1]) * S + (w[:, None] * Xd).T @ Bc
    return y


def test_p4_ssd_materialised_and_s6_equivalence():
    inp = ssd_inputs(2, 19, 4, 3, 5, ngroups=2, seed=7, bf16=False, with_z=True)
    y, fs = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["z"], inp["delta_bias"], return_final_state=True)
    ref = materialised_ssd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["z"], inp["delta_bias"])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)
    # the same problem as an S6 scan with channels d = (head, p), Delta and A shared per head
    batch, L, H, P = inp["x"].shape
    G, N = inp["B"].shape[2], inp["B"].shape[3]
    for g in range(G):
        heads = range(g * (H // G), (g + 1) * (H // G))
        u = np.concatenate([inp["x"][:, :, h, :].transpose(0, 2, 1) for h in heads], axis=1)
        dl = np.concatenate([np.repeat(inp["delta"][:, None, :, h], P, axis=1) for h in heads], axis=1)
        zz = np.concatenate([inp["z"][:, :, h, :].transpose(0, 2, 1) for h in heads], axis=1)
        A6 = np.concatenate([np.full((P, N), inp["A"][h]) for h in heads], axis=0)
        D6 = np.concatenate([np.full(P, inp["D"][h]) for h in heads])
        b6 = np.concatenate([np.full(P, inp["delta_bias"][h]) for h in heads])
        B6 = inp["B"][:, :, g, :].transpose(0, 2, 1)
        C6 = inp["C"][:, :, g, :].transpose(0, 2, 1)
        y6, h6 = oracle.s6_fwd(u, dl, A6, B6, C6, D6, zz, b6, return_last_state=True)
        for i, h in enumerate(heads):
            np.testing.assert_allclose(y[:, :, h, :], y6[:, i * P:(i + 1) * P, :].transpose(0, 2, 1),
                                       rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(fs[:, h], h6[:, i * P:(i + 1) * P, :], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("Q", [4, 8])
def test_p4_ssd_chunked_decomposition(Q):
    inp = ssd_inputs(1, 21, 2, 3, 6, ngroups=1, seed=9, bf16=False)
    y = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                       None, inp["delta_bias"])
    ref = chunked_ssd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], Q, inp["D"],
                      inp["delta_bias"])
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------- P5
def _fd_check(inp, with_z=True, with_D=True, with_bias=True, eps=1e-6):
    rng = np.random.default_rng(21)
    keys = ["u", "delta", "A", "B", "C"] + (["D"] if with_D else []) + \
           (["z"] if with_z else []) + (["delta_bias"] if with_bias else [])
    base = {k: (None if inp.get(k) is None else np.asarray(inp[k], np.float64).copy())
            for k in ["u", "delta", "A", "B", "C", "D", "z", "delta_bias"]}
    if not with_z:
        base["z"] = None
    if not with_D:
        base["D"] = None
    if not with_bias:
        base["delta_bias"] = None
    y0 = oracle.s6_fwd(**{k: base[k] for k in base})
    w = rng.standard_normal(y0.shape)
    g = oracle.s6_bwd(dy=w, **{k: base[k] for k in base})
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    for k in keys:
        arr = base[k]
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + eps
            fp = np.sum(w * oracle.s6_fwd(**base))
            arr[idx] = old - eps
            fm = np.sum(w * oracle.s6_fwd(**base))
            arr[idx] = old
            fd[idx] = (fp - fm) / (2 * eps)
        an = g[names[k]]
        scale = np.max(np.abs(fd)) + 1e-30
        assert np.max(np.abs(an - fd)) <= 1e-6 * max(scale, 1.0), (k, np.max(np.abs(an - fd)), scale)


def test_p5_finite_differences_full():
    _fd_check(s6_inputs(2, 4, 16, 4, seed=13))


def test_p5_finite_differences_no_gate_no_D():
    _fd_check(s6_inputs(1, 3, 12, 3, seed=17), with_z=False, with_D=False, with_bias=False)


def test_p5_finite_differences_config0_size():
    # tiny configuration size (1 x 4 x 64, N = 16), gradients w.r.t. the shared B, C and A
    inp = s6_inputs(1, 4, 64, 16, seed=160_000)
    rng = np.random.default_rng(3)
    base = {k: (None if v is None else np.asarray(v, np.float64).copy()) for k, v in inp.items()
            if k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    y0 = oracle.s6_fwd(**base)
    w = rng.standard_normal(y0.shape)
    g = oracle.s6_bwd(dy=w, **base)
    eps = 1e-6
    for key, gname in (("B", "dB"), ("C", "dC"), ("A", "dA"), ("delta", "ddelta")):
        arr = base[key]
        for idx in [tuple(rng.integers(0, s) for s in arr.shape) for _ in range(12)]:
            old = arr[idx]
            arr[idx] = old + eps
            fp = np.sum(w * oracle.s6_fwd(**base))
            arr[idx] = old - eps
            fm = np.sum(w * oracle.s6_fwd(**base))
            arr[idx] = old
            fd = (fp - fm) / (2 * eps)
            assert abs(g[gname][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (key, idx, g[gname][idx], fd)


# ----------------------------------------------------------------------------- P6
def test_p6_linearity_in_u(tiny):
    inp = tiny
    rng = np.random.default_rng(1)
    u2 = rng.standard_normal(inp["u"].shape)
    args = dict(delta=inp["delta"], A=inp["A"], B=inp["B"], C=inp["C"], D=inp["D"],
                z=inp["z"], delta_bias=inp["delta_bias"])
    y1 = oracle.s6_fwd(inp["u"], **args)
    y2 = oracle.s6_fwd(u2, **args)
    y12 = oracle.s6_fwd(1.5 * inp["u"].astype(np.float64) - 0.25 * u2, **args)
    np.testing.assert_allclose(y12, 1.5 * y1 - 0.25 * y2, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("k", [1, 7, 23])
def test_p6_split_scan(tiny, k):
    inp = tiny
    L = inp["u"].shape[2]
    args = dict(A=inp["A"], D=inp["D"], delta_bias=inp["delta_bias"])
    y, hl = oracle.s6_fwd(inp["u"], inp["delta"], B=inp["B"], C=inp["C"], z=inp["z"],
                          return_last_state=True, **args)
    ya, ha = oracle.s6_fwd(inp["u"][:, :, :k], inp["delta"][:, :, :k], B=inp["B"][:, :, :k],
                           C=inp["C"][:, :, :k], z=inp["z"][:, :, :k], return_last_state=True, **args)
    yb, hb = oracle.s6_fwd(inp["u"][:, :, k:], inp["delta"][:, :, k:], B=inp["B"][:, :, k:],
                           C=inp["C"][:, :, k:], z=inp["z"][:, :, k:], h0=ha,
                           return_last_state=True, **args)
    np.testing.assert_allclose(np.concatenate([ya, yb], axis=2), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hb, hl, rtol=1e-12, atol=1e-13)
    assert y.shape[2] == L


# ----------------------------------------------------------------------------- P7
def test_p7_decay_bound():
    inp = s6_inputs(2, 6, 200, 16, seed=19)
    y, hl = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["z"], inp["delta_bias"], return_last_state=True)
    dt = softplus(inp["delta"].astype(np.float64) + inp["delta_bias"][None, :, None])
    # |h_L,n| <= sum_s |Delta_s B_sn u_s|
    bound = np.einsum("bdl,bnl->bdn", np.abs(dt * inp["u"]), np.abs(inp["B"].astype(np.float64)))
    assert np.all(np.abs(hl) <= bound * (1 + 1e-12))
    assert np.all(np.isfinite(y))


# ----------------------------------------------------------------------------- P8
def test_p8_single_step():
    rng = np.random.default_rng(2)
    N = 16
    u = rng.standard_normal((1, 1, 1))
    delta = rng.standard_normal((1, 1, 1))
    z = rng.standard_normal((1, 1, 1))
    B = rng.standard_normal((1, N, 1))
    C = rng.standard_normal((1, N, 1))
    A = -np.arange(1.0, N + 1)[None, :]
    D = np.array([0.7])
    bias = np.array([-1.3])
    y = oracle.s6_fwd(u, delta, A, B, C, D, z, bias)
    dt = np.log1p(np.exp(delta[0, 0, 0] + bias[0]))
    hand = (np.dot(C[0, :, 0], dt * B[0, :, 0] * u[0, 0, 0]) + D[0] * u[0, 0, 0]) \
        * z[0, 0, 0] / (1.0 + np.exp(-z[0, 0, 0]))
    assert abs(y[0, 0, 0] - hand) <= 1e-14 * (1 + abs(hand))


def test_p8_study_note_three_steps():
    # The study note's one-step pseudocode: h_t = exp(-Delta) h_{t-1} + Delta B x_t,
    # y_t = C h_t, i.e. N = 1, A = -1, no D and no gate.  Delta_t = softplus(delta_t).
    x = np.array([1.0, -2.0, 0.5])
    dl = np.array([0.0, 1.0, -1.0])
    Bv = np.array([2.0, 1.0, -1.0])
    Cv = np.array([1.0, 3.0, 2.0])
    y = oracle.s6_fwd(x[None, None], dl[None, None], np.array([[-1.0]]), Bv[None, None],
                      Cv[None, None])
    D0, D1, D2 = np.log(2.0), np.log(1 + np.e), np.log(1 + 1 / np.e)
    h0 = D0 * 2.0 * 1.0
    h1 = np.exp(-D1) * h0 + D1 * 1.0 * -2.0
    h2 = np.exp(-D2) * h1 + D2 * -1.0 * 0.5
    np.testing.assert_allclose(y[0, 0], [1.0 * h0, 3.0 * h1, 2.0 * h2], rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------- P9
@pytest.mark.parametrize("with_z,with_D,with_bias", [(True, True, True), (False, False, False)])
def test_p9_decode_steps_equal_scan(with_z, with_D, with_bias):
    """The decode-step oracle run token by token from a state equals the scan
    over the same tokens from that state (recurrent mode = scan mode)."""
    inp = s6_inputs(2, 5, 9, 16, seed=41, with_z=with_z, with_D=with_D, with_bias=with_bias)
    rng = np.random.default_rng(5)
    h0 = rng.standard_normal((2, 5, 16))
    y_scan, h_scan = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                   inp["delta_bias"], h0=h0, return_last_state=True)
    h = h0
    ys = []
    for t in range(9):
        zt = None if inp["z"] is None else inp["z"][:, :, t]
        y, h = oracle.s6_step(inp["u"][:, :, t], inp["delta"][:, :, t], inp["A"], inp["B"][:, :, t],
                              inp["C"][:, :, t], inp["D"], zt, inp["delta_bias"], h)
        ys.append(y)
    np.testing.assert_allclose(np.stack(ys, axis=2), y_scan, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h, h_scan, rtol=1e-12, atol=1e-13)


def test_p9_decode_step_from_zero_is_first_scan_step():
    inp = s6_inputs(1, 3, 4, 8, seed=42)
    y_scan = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                           inp["delta_bias"])
    y, h = oracle.s6_step(inp["u"][:, :, 0], inp["delta"][:, :, 0], inp["A"], inp["B"][:, :, 0],
                          inp["C"][:, :, 0], inp["D"], inp["z"][:, :, 0], inp["delta_bias"])
    np.testing.assert_allclose(y, y_scan[:, :, 0], rtol=1e-13, atol=1e-14)
    assert h.shape == (1, 3, 8)


# ---------------------------------------------------------------------------- P10
@pytest.mark.parametrize("K", [1, 3, 4, 8])
def test_p10_conv1d_is_numpy_convolve(K):
    """Without the activation the causal conv of every channel is numpy's full
    convolution with the reversed kernel, first L outputs, plus the bias."""
    rng = np.random.default_rng(60 + K)
    x = rng.standard_normal((2, 3, 37))
    w = rng.standard_normal((3, K))
    bias = rng.standard_normal(3)
    out = oracle.causal_conv1d(x, w, bias, silu=False)
    for b in range(2):
        for d in range(3):
            ref = np.convolve(x[b, d], w[d][::-1])[:37] + bias[d]
            np.testing.assert_allclose(out[b, d], ref, rtol=1e-13, atol=1e-13)


def test_p10_conv1d_causal_and_silu():
    rng = np.random.default_rng(70)
    x = rng.standard_normal((1, 4, 20))
    w = rng.standard_normal((4, 4))
    y0 = oracle.causal_conv1d(x, w)
    x2 = x.copy()
    x2[:, :, 11] += 5.0
    y1 = oracle.causal_conv1d(x2, w)
    np.testing.assert_array_equal(y0[:, :, :11], y1[:, :, :11])       # no output before the change moves
    assert np.all(y0[:, :, 11] != y1[:, :, 11])
    pre = oracle.causal_conv1d(x, w, silu=False)
    np.testing.assert_allclose(y0, pre * 0.5 * (1.0 + np.tanh(0.5 * pre)), rtol=1e-13, atol=1e-15)


def test_p10_conv1d_update_chain_equals_sequence():
    rng = np.random.default_rng(71)
    x = rng.standard_normal((2, 5, 12))
    w = rng.standard_normal((5, 4))
    bias = rng.standard_normal(5)
    ref = oracle.causal_conv1d(x, w, bias)
    state = np.zeros((2, 5, 3))
    outs = []
    for t in range(12):
        o, state = oracle.causal_conv1d_update(x[:, :, t], state, w, bias)
        outs.append(o)
    np.testing.assert_allclose(np.stack(outs, axis=2), ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(state, x[:, :, -3:])


@pytest.mark.parametrize("K,silu", [(4, True), (3, False), (1, True)])
def test_p10_conv1d_backward_finite_differences(K, silu):
    """The conv backward against central finite differences of <dout, out> of
    the conv oracle, for every entry of x, the weights and the bias."""
    rng = np.random.default_rng(72 + K)
    x = rng.standard_normal((2, 3, 9))
    w = rng.standard_normal((3, K))
    bias = rng.standard_normal(3)
    dout = rng.standard_normal((2, 3, 9))
    dx, dw, db = oracle.causal_conv1d_bwd(x, w, bias, dout, silu=silu)
    h = 1e-6

    def loss(x_, w_, b_):
        return float((oracle.causal_conv1d(x_, w_, b_, silu=silu) * dout).sum())
    for arr, grad in ((x, dx), (w, dw), (bias, db)):
        num = np.empty_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(x, w, bias)
            arr[idx] = old - h
            lm = loss(x, w, bias)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7)


# ---------------------------------------------------------------------------- P11
def _delta_for(dt):
    """pre-activation delta whose softplus is dt (bias 0)"""
    return np.log(np.expm1(np.asarray(dt, np.float64)))


def test_p11_zoh_is_the_exact_held_input_step():
    """Zero-order hold: with u, B held over each step, the discrete state equals
    the continuous system dh/ds = A h + B u integrated by scipy's ODE solver."""
    from scipy.integrate import solve_ivp
    rng = np.random.default_rng(80)
    N, L = 3, 5
    A = np.array([[-0.5, -2.0, -7.0]])
    dts = rng.uniform(0.05, 0.4, L)
    u = rng.standard_normal(L)
    B = rng.standard_normal((N, L))
    C = rng.standard_normal((N, L))
    h0 = rng.standard_normal(N)
    y, hl = oracle.s6_fwd_disc(oracle.DISC_ZOH, u[None, None], _delta_for(dts)[None, None], A, B[None],
                               C[None], h0=h0[None, None], return_last_state=True)
    h = h0.copy()
    for t in range(L):
        sol = solve_ivp(lambda s, v: A[0] * v + B[:, t] * u[t], (0.0, dts[t]), h, rtol=1e-12, atol=1e-14,
                        method="DOP853")
        h = sol.y[:, -1]
        assert abs(y[0, 0, t] - np.dot(C[:, t], h)) <= 1e-9 * (1 + abs(y[0, 0, t]))
    np.testing.assert_allclose(hl[0, 0], h, rtol=1e-9, atol=1e-12)


def test_p11_zoh_tends_to_euler_as_a_vanishes():
    inp = s6_inputs(1, 3, 20, 4, seed=81)
    A = np.full((3, 4), -1e-9)
    args = (inp["u"], inp["delta"], A, inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])
    np.testing.assert_allclose(oracle.s6_fwd_disc(oracle.DISC_ZOH, *args), oracle.s6_fwd(*args),
                               rtol=1e-7, atol=1e-9)


# ---------------------------------------------------------------------------- P12
def _order_study(disc, steps):
    """error at s = 2 of the discretised dh/ds = -1.3 h + 0.7 (1 - cos s), h(0) = 0,
    sampled at s_t = t * 2 / steps (the input vanishes before s = 0)"""
    from scipy.integrate import solve_ivp
    exact = solve_ivp(lambda s, v: -1.3 * v + 0.7 * (1 - np.cos(s)), (0.0, 2.0), [0.0], rtol=1e-13,
                      atol=1e-15, method="DOP853").y[0, -1]
    errs = []
    for T in steps:
        dt = 2.0 / T
        s_t = dt * np.arange(T + 1)
        L = T + 1
        y = oracle.s6_fwd_disc(disc, (1 - np.cos(s_t))[None, None], np.full((1, 1, L), _delta_for(dt)),
                               np.array([[-1.3]]), np.full((1, 1, L), 0.7), np.ones((1, 1, L)))
        errs.append(abs(y[0, 0, -1] - exact))
    return errs


def test_p12_trapezoid_is_second_order_euler_first_order():
    """The exponential-trapezoidal input rule (Mamba 解密 sec. 6.3) converges with
    order 2 in the step, the exponential-Euler rule with order 1."""
    steps = (50, 100, 200, 400)
    et = _order_study(oracle.DISC_TRAPEZOID, steps)
    ee = _order_study(oracle.DISC_EULER, steps)
    for a, b in zip(et, et[1:]):
        assert 3.7 < a / b < 4.3, et
    for a, b in zip(ee, ee[1:]):
        assert 1.8 < a / b < 2.2, ee
    assert et[-1] < ee[-1] / 100


def test_p12_trapezoid_constant_input_steady_state():
    """Constant Delta, B, u: the trapezoidal state tends to the fixed point
    h* = (1/2) Delta B u (1 + abar) / (1 - abar)."""
    dt, A, Bv, uv, L = 0.1, -2.0, 0.6, 1.5, 400
    y, hl = oracle.s6_fwd_disc(oracle.DISC_TRAPEZOID, np.full((1, 1, L), uv), np.full((1, 1, L), _delta_for(dt)),
                               np.array([[A]]), np.full((1, 1, L), Bv), np.ones((1, 1, L)),
                               return_last_state=True)
    ab = np.exp(dt * A)
    assert abs(hl[0, 0, 0] - 0.5 * dt * Bv * uv * (1 + ab) / (1 - ab)) < 1e-12


# ---------------------------------------------------------------------------- P13
def test_p13_ssd_backward_finite_differences():
    """The SSD backward (built on the S6 backward through the channel mapping
    of P4) against central finite differences of <dy, y> of the SSD forward
    oracle, for every entry of every input (2 groups, all optional inputs)."""
    inp = ssd_inputs(1, 7, 4, 2, 3, ngroups=2, seed=91, bf16=False, with_z=True)
    dy = np.random.default_rng(92).standard_normal(inp["x"].shape)
    keys = ("x", "delta", "A", "B", "C", "D", "z", "delta_bias")
    base = {k: np.array(inp[k], dtype=np.float64) for k in keys}
    g = oracle.ssd_bwd(*(base[k] for k in keys), dy=dy)

    def loss(v):
        return float((oracle.ssd_fwd(*(v[k] for k in keys)) * dy).sum())

    names = {"x": "dx", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
             "delta_bias": "ddelta_bias"}
    eps = 1e-6
    for k in keys:
        for idx in np.ndindex(base[k].shape):
            vp = dict(base); vp[k] = base[k].copy(); vp[k][idx] += eps
            vm = dict(base); vm[k] = base[k].copy(); vm[k][idx] -= eps
            fd = (loss(vp) - loss(vm)) / (2 * eps)
            assert abs(g[names[k]][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (k, idx, g[names[k]][idx], fd)


# ------------------------------------------------------------------ planted mistakes
MUTATIONS = [
    # (description, original text, mutated text)
    ("drop the input term", "+ dt * B[n * L + t] * u[t];\n            acc",
     ";\n            acc"),
    ("wrong sign of A", "double abar = exp(dt * A[n]);\n            h[n]",
     "double abar = exp(-dt * A[n]);\n            h[n]"),
    ("B and C swapped", "acc += C[n * L + t] * h[n];", "acc += B[n * L + t] * h[n];"),
    ("drop D feed-through", "acc += D * u[t];\n        if (z) acc *= z[t] * sigmoid_d(z[t]);",
     "if (z) acc *= z[t] * sigmoid_d(z[t]);"),
    ("gate by sigmoid only", "if (z) acc *= z[t] * sigmoid_d(z[t]);", "if (z) acc *= sigmoid_d(z[t]);"),
    ("bwd: lambda without decay", "double l = gp * C[n * L + t] + abar_next * lam[n];",
     "double l = gp * C[n * L + t] + lam[n];"),
    ("bwd: dA uses h_t", "dA_row[n] += l * dt * abar * hprev;",
     "dA_row[n] += l * dt * abar * hs[(t + 1) * N + n];"),
    ("ssd: decay index off by one", "double hv = a * H[p * N + n] + dt * xp * B[t * sb + n];",
     "double hv = a * H[p * N + n] + dt * xp * B[(t > 0 ? t - 1 : t) * sb + n];"),
    ("zoh: divided by Delta A instead of A", "in = (A[n] != 0.0 ? expm1(dt * A[n]) / A[n] : dt) * bu;",
     "in = (A[n] != 0.0 ? expm1(dt * A[n]) / (dt * A[n]) : dt) * bu;"),
    ("trapezoid: previous term without decay", "in = 0.5 * (e + abar * eprev[n]);",
     "in = 0.5 * (e + eprev[n]);"),
    ("trapezoid: no halving", "in = 0.5 * (e + abar * eprev[n]);", "in = e + abar * eprev[n];"),
    ("softplus: wrong sign inside log1p", "return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));",
     "return (x > 0.0 ? x : 0.0) + log1p(exp(fabs(x)));"),
    ("fwd: Delta_bias not added", "double dt = softplus_d(delta[t] + bias);\n        double acc = 0.0;",
     "double dt = softplus_d(delta[t]);\n        double acc = 0.0;"),
    ("bwd: ddelta without the softplus derivative", "ddelta[t] = dDelta * sigmoid_d(x);",
     "ddelta[t] = dDelta;"),
    ("bwd: dDelta without the decay term", "dDelta += l * (B[n * L + t] * u[t] + A[n] * abar * hprev);",
     "dDelta += l * B[n * L + t] * u[t];"),
    ("ssd: heads mapped to groups round-robin", "g = h / hpg;", "g = h % ngroups;"),
    ("ssd: every channel of a head driven by its first", "dt * xp * B[t * sb + n]", "dt * x[t * sx] * B[t * sb + n]"),
    ("ssd: D feed-through dropped", "acc += D * xp;\n            if (z) {", "if (z) {"),
]


@pytest.mark.parametrize("desc,orig,mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes(tmp_path, desc, orig, mut, monkeypatch):
    """Plant each mistake in a CPU copy of the oracle and check a pin catches it."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "msc_oracle.c")).read()
    assert orig in src, desc
    bad = tmp_path / "bad.c"
    bad.write_text(src.replace(orig, mut, 1))
    so = tmp_path / "libbad.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(bad), "-lm"],
                   check=True)
    monkeypatch.setattr(oracle, "_LIB", str(so))
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    monkeypatch.setattr(oracle, "_lib", None)
    caught = False
    for pin in (lambda: test_p1_closed_form(True, True, True),
                lambda: test_p5_finite_differences_full(),
                lambda: test_p4_ssd_materialised_and_s6_equivalence(),
                lambda: test_p11_zoh_is_the_exact_held_input_step(),
                lambda: test_p12_trapezoid_is_second_order_euler_first_order(),
                lambda: test_p12_trapezoid_constant_input_steady_state()):
        try:
            pin()
        except AssertionError:
            caught = True
            break
    monkeypatch.setattr(oracle, "_lib", None)
    assert caught, "no pin caught: " + desc


PY_MUTATIONS = [
    # (description, function, original text, mutated text, pin) in oracle.py
    ("conv bwd: taps not reversed", "causal_conv1d_bwd", "gp[:, :, K - 1 - k:K - 1 - k + L]", "gp[:, :, k:k + L]",
     "p10"),
    ("conv bwd: silu derivative without its second term", "causal_conv1d_bwd",
     "g = g * sg * (1.0 + pre * (1.0 - sg))", "g = g * sg", "p10"),
    ("ssd bwd: B of the first group for every group", "ssd_bwd",
     "B[:, :, g, :].transpose(0, 2, 1), C[:, :, g, :]", "B[:, :, 0, :].transpose(0, 2, 1), C[:, :, g, :]", "p13"),
    ("ssd bwd: ddelta from one channel of the head", "ssd_bwd",
     'r["ddelta"][:, sl, :].sum(axis=1)', 'r["ddelta"][:, i * P, :]', "p13"),
    ("ssd bwd: dA from one channel of the head", "ssd_bwd", 'r["dA"][sl].sum()', 'r["dA"][sl][0].sum()', "p13"),
    ("ssd bwd: dx of the group's first head for every head", "ssd_bwd",
     'r["du"][:, sl, :]', 'r["du"][:, :P, :]', "p13"),
    ("conv: taps in reverse order", "causal_conv1d", "out += w[None, :, k, None] * xp[:, :, k:k + L]",
     "out += w[None, :, K - 1 - k, None] * xp[:, :, k:k + L]", "p10_fwd"),
    ("conv decode step: state not shifted", "causal_conv1d_update", "window[:, :, 1:]", "window[:, :, :-1]",
     "p10_update"),
    ("decode step: gate dropped", "s6_step", "z = None if z is None else _f64(z)[:, :, None]", "z = None", "p9"),
]

PY_PINS = {
    "p9": lambda: test_p9_decode_steps_equal_scan(True, True, True),
    "p10": lambda: test_p10_conv1d_backward_finite_differences(4, True),
    "p10_fwd": lambda: test_p10_conv1d_is_numpy_convolve(4),
    "p10_update": lambda: test_p10_conv1d_update_chain_equals_sequence(),
    "p13": lambda: test_p13_ssd_backward_finite_differences(),
}


@pytest.mark.parametrize("desc,fn,orig,mut,pin", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_planted_mistakes_python(desc, fn, orig, mut, pin, monkeypatch):
    """Plant each mistake in a copy of a Python oracle function and check that
    its pin fails."""
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn)))
    assert orig in src, desc
    ns = dict(vars(oracle))
    exec(compile(src.replace(orig, mut, 1), "<planted>", "exec"), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    with pytest.raises(AssertionError):
        PY_PINS[pin]()
