"""GPU parity of the S6 forward with the causal conv1d + SiLU front end fused
into the scan (msc_selective_scan_fwd_conv, through the C ABI) against the
oracle's conv1d followed by its scan, u kept in double precision (the fused
kernel keeps u in fp32, never rounding it to the input dtype).  Rows of any
length: the TMA kernel takes rows it can stream, the plain-load kernel the
rest.

Tolerances (max |gpu - ref| / (1 + |ref|)) as the S6 forward: 1e-4 with fp32
inputs, 2e-3 with bf16 inputs (the oracle consumes the same bf16-rounded x)."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, conv_taps
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-3


def _run(inp, w, cb, bf16, h0=None, last=False):
    import selective_state_space_160_b300 as msc
    dev = {k: to_dev(inp[k], bf16) for k in ("u", "delta", "z", "B", "C")}
    out = msc.msc_selective_scan_fwd_conv(
        dev["u"], to_dev(w), to_dev(cb), dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
        to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]),
        h0=to_dev(h0) if h0 is not None else None, return_last_state=last)
    if last:
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy()


def _ref(inp, w, cb, h0=None, last=False):
    u = oracle.causal_conv1d(inp["u"], w, cb)
    return oracle.s6_fwd(u, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"],
                         h0=h0, return_last_state=last)


@pytest.mark.parametrize("batch,dim,L,N,K,bf16", [
    (1, 4, 64, 16, 4, False), (2, 37, 96, 16, 4, True), (2, 40, 1000, 16, 3, True),
    (1, 33, 256, 4, 2, False), (3, 8, 64, 16, 1, True), (1, 70, 104, 16, 4, True), (2, 5, 36, 7, 4, False)])
def test_shapes(batch, dim, L, N, K, bf16):
    inp = s6_inputs(batch, dim, L, N, seed=4000 + batch + dim + L + N + K, bf16=bf16)
    w, cb = conv_taps(dim, K, seed=4100 + K)
    y = _run(inp, w, cb, bf16)
    assert max_rel_err(y, _ref(inp, w, cb)) <= (TOL_BF16 if bf16 else TOL_F32)


def test_optional_inputs_and_states():
    inp = s6_inputs(2, 36, 128, 16, seed=4200, with_z=False, with_D=False, with_bias=False)
    w, _ = conv_taps(36, 4, seed=4201)
    y = _run(inp, w, None, False)
    assert max_rel_err(y, _ref(inp, w, None)) <= TOL_F32
    inp = s6_inputs(2, 36, 128, 16, seed=4202, bf16=True)
    w, cb = conv_taps(36, 4, seed=4203)
    h0 = np.random.default_rng(4204).standard_normal((2, 36, 16)).astype(np.float32)
    y, hl = _run(inp, w, cb, True, h0=h0, last=True)
    ry, rhl = _ref(inp, w, cb, h0=h0, last=True)
    assert max_rel_err(y, ry) <= TOL_BF16
    assert max_rel_err(hl, rhl) <= TOL_BF16


def test_long_sequence_segments():
    """Few rows and a long sequence: the row is split into segments, and every
    segment reads the conv's three-step halo of the previous one from memory."""
    inp = s6_inputs(1, 48, 16384, 16, seed=4300, bf16=True)
    w, cb = conv_taps(48, 4, seed=4301)
    y, hl = _run(inp, w, cb, True, last=True)
    ry, rhl = _ref(inp, w, cb, last=True)
    assert max_rel_err(y, ry) <= TOL_BF16
    assert max_rel_err(hl, rhl) <= TOL_BF16


def test_equals_two_launches_fp32():
    """fp32 inputs: the fused call equals msc_causal_conv1d_fwd (fp32 out)
    followed by msc_selective_scan_fwd, up to fp32 rounding."""
    import selective_state_space_160_b300 as msc
    inp = s6_inputs(2, 64, 512, 16, seed=4400)
    w, cb = conv_taps(64, 4, seed=4401)
    y = _run(inp, w, cb, False)
    u = msc.msc_causal_conv1d_fwd(to_dev(inp["u"]), to_dev(w), to_dev(cb))
    y2 = msc.msc_selective_scan_fwd(u, to_dev(inp["delta"]), to_dev(inp["A"]), to_dev(inp["B"]), to_dev(inp["C"]),
                                    to_dev(inp["D"]), to_dev(inp["z"]), to_dev(inp["delta_bias"])).cpu().numpy()
    assert max_rel_err(y, y2) <= 1e-5


def test_mamba_layer_size_sampled_rows():
    """The launch the bench times (batch 8, D 5120, L 2048, N 16, bf16, K 4),
    oracle on every 37th channel of every batch entry."""
    inp = s6_inputs(8, 5120, 2048, 16, seed=4500, bf16=True)
    w, cb = conv_taps(5120, 4, seed=4501)
    y = _run(inp, w, cb, True)
    assert np.all(np.isfinite(y))
    ds = np.arange(0, 5120, 37)
    sub = dict(inp)
    for k in ("u", "delta", "z"):
        sub[k] = inp[k][:, ds, :]
    sub["A"] = inp["A"][ds]
    for k in ("D", "delta_bias"):
        sub[k] = inp[k][ds]
    assert max_rel_err(y[:, ds, :], _ref(sub, w[ds], cb[ds])) <= TOL_BF16


@pytest.mark.parametrize("batch,dim,L,N,K,bf16", [
    (1, 4, 100, 16, 4, True), (2, 37, 1, 16, 4, True), (1, 33, 3, 5, 3, False), (2, 40, 1031, 16, 4, False),
    (3, 65, 257, 16, 2, True), (1, 9, 7, 1, 1, True)])
def test_unaligned_rows(batch, dim, L, N, K, bf16):
    """Rows TMA cannot stream as they are (seqlen not a multiple of 8 with bf16
    inputs, of 4 with fp32): the plain-load kernel forms the conv step by step,
    the first three steps reading zeros before t = 0."""
    inp = s6_inputs(batch, dim, L, N, seed=4700 + batch + dim + L + N + K, bf16=bf16)
    w, cb = conv_taps(dim, K, seed=4701 + K)
    h0 = np.random.default_rng(4702).standard_normal((batch, dim, N)).astype(np.float32)
    y, hl = _run(inp, w, cb, bf16, h0=h0, last=True)
    ry, rhl = _ref(inp, w, cb, h0=h0, last=True)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y, ry) <= tol
    assert max_rel_err(hl, rhl) <= tol


def test_unaligned_rows_segments():
    """Few rows and a long, unaligned sequence: the plain-load kernel's segments
    each read the conv's three-step halo of the previous segment from memory."""
    inp = s6_inputs(1, 20, 9001, 16, seed=4800, bf16=True)
    w, cb = conv_taps(20, 4, seed=4801)
    y, hl = _run(inp, w, cb, True, last=True)
    ry, rhl = _ref(inp, w, cb, last=True)
    assert max_rel_err(y, ry) <= TOL_BF16
    assert max_rel_err(hl, rhl) <= TOL_BF16


@pytest.mark.parametrize("batch,dim,L,bf16", [(2, 37, 96, True), (1, 24, 2048, False)])
def test_plain_kernel_agrees_with_tma_kernel(monkeypatch, batch, dim, L, bf16):
    """On rows both kernels take, the plain-load kernel (forced by
    MSC_S6_FWD_PLAIN) and the TMA kernel agree to fp32 rounding."""
    inp = s6_inputs(batch, dim, L, 16, seed=4900 + L, bf16=bf16)
    w, cb = conv_taps(dim, 4, seed=4901)
    y_tma = _run(inp, w, cb, bf16)
    monkeypatch.setenv("MSC_S6_FWD_PLAIN", "1")
    y_plain = _run(inp, w, cb, bf16)
    assert max_rel_err(y_plain, y_tma) <= 1e-5
