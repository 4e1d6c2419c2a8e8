"""GPU parity of the causal conv1d front end and its decode step (through the C
ABI) against the oracle.

Tolerances: with an fp32 output max |gpu - ref| / (1 + |ref|) <= 1e-4.  A bf16
output is a quantised value (8 significant bits, up to 2^-8 relative rounding
error), so both sides take the same quantisation: the GPU value must equal the
oracle's value rounded to bf16, or its neighbour one bf16 ulp away when the
fp32 result before rounding lies within rounding distance of a boundary, and
an output that nearly cancels to zero may differ by the fp32 accumulation
error of its sum (see bf16_match).  The
oracle consumes the same bf16-rounded inputs."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import bf16_round
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu


def _data(batch, dim, L, K, seed, bf16):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, dim, L)).astype(np.float32)
    if bf16:
        x = bf16_round(x)
    w = (rng.standard_normal((dim, K)) / np.sqrt(K)).astype(np.float32)
    bias = (0.1 * rng.standard_normal(dim)).astype(np.float32)
    return x, w, bias


def _out_np(t):
    return t.float().cpu().numpy()


def bf16_match(got, ref, x, w, bias):
    """Largest |got - bf16(ref)| over its allowance (<= 1 passes).  The allowance
    is one bf16 ulp at |ref| plus the fp32 accumulation error of the sum
    before the activation, 2^-20 (|bias| + sum_k |w_k x|): an output that nearly
    cancels to zero has a bf16 ulp far below what fp32 arithmetic resolves."""
    r = bf16_round(np.asarray(ref, np.float32)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -120))) - 7)
    mag = oracle.causal_conv1d(np.abs(x), np.abs(w), None if bias is None else np.abs(bias), silu=False)
    return float(np.max(np.abs(np.asarray(got, np.float64) - r) / (ulp + 2.0 ** -20 * mag)))


@pytest.mark.parametrize("batch,dim,L,K", [(1, 4, 64, 4), (2, 37, 100, 4), (3, 5, 7, 3), (1, 70, 1, 4),
                                           (2, 16, 256, 8), (1, 9, 33, 1), (2, 12, 40, 2)])
@pytest.mark.parametrize("in_bf16,out_bf16", [(False, False), (True, False), (True, True)])
def test_forward_shapes(batch, dim, L, K, in_bf16, out_bf16):
    import torch
    import selective_state_space_160_b300 as msc
    x, w, bias = _data(batch, dim, L, K, 900 + batch + dim + L + K, in_bf16)
    out = msc.msc_causal_conv1d_fwd(to_dev(x, in_bf16), to_dev(w), to_dev(bias),
                                    out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    ref = oracle.causal_conv1d(x, w, bias)
    if out_bf16:
        assert bf16_match(_out_np(out), ref, x, w, bias) <= 1.0
    else:
        assert max_rel_err(_out_np(out), ref) <= 1e-4


@pytest.mark.parametrize("batch,dim,L,K", [(2, 40, 1048, 4), (3, 7, 2048, 3), (1, 30, 520, 4), (1, 3, 8, 4),
                                           (4, 700, 1024, 4)])
@pytest.mark.parametrize("in_bf16,out_bf16", [(False, True), (True, True), (False, False)])
def test_forward_long_rows(batch, dim, L, K, in_bf16, out_bf16):
    """Rows of several 512-step units, a partial last unit ending in an 8-step
    lane, and (4 x 700 rows x 2 units) more units than one sweep of the grid."""
    import torch
    import selective_state_space_160_b300 as msc
    x, w, bias = _data(batch, dim, L, K, 970 + batch + dim + L + K, in_bf16)
    out = msc.msc_causal_conv1d_fwd(to_dev(x, in_bf16), to_dev(w), to_dev(bias),
                                    out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    ref = oracle.causal_conv1d(x, w, bias)
    if out_bf16:
        assert bf16_match(_out_np(out), ref, x, w, bias) <= 1.0
    else:
        assert max_rel_err(_out_np(out), ref) <= 1e-4


@pytest.mark.parametrize("silu,with_bias", [(False, True), (True, False), (False, False)])
def test_forward_options(silu, with_bias):
    import selective_state_space_160_b300 as msc
    x, w, bias = _data(2, 24, 64, 4, 950, False)
    b = bias if with_bias else None
    out = msc.msc_causal_conv1d_fwd(to_dev(x), to_dev(w), to_dev(b), silu=silu)
    assert max_rel_err(_out_np(out), oracle.causal_conv1d(x, w, b, silu=silu)) <= 1e-4


@pytest.mark.parametrize("K", [4, 1, 6])
def test_update_chain_matches_forward(K):
    """Decode steps from a zero state reproduce the sequence convolution and
    leave the last K - 1 inputs in the state."""
    import torch
    import selective_state_space_160_b300 as msc
    x, w, bias = _data(2, 33, 20, K, 960 + K, True)
    state = torch.zeros((2, 33, K - 1), dtype=torch.float32, device="cuda")
    outs = []
    for t in range(20):
        o = msc.msc_causal_conv1d_update(to_dev(np.ascontiguousarray(x[:, :, t]), True), state, to_dev(w),
                                         to_dev(bias), out_dtype=torch.float32)
        outs.append(_out_np(o))
    ref = oracle.causal_conv1d(x, w, bias)
    assert max_rel_err(np.stack(outs, axis=2), ref) <= 1e-4
    if K > 1:
        np.testing.assert_array_equal(state.cpu().numpy(), x[:, :, 20 - (K - 1):])


def test_feeds_the_scan():
    """conv1d (bf16 out) -> S6 forward equals the oracle chain on the same values."""
    import torch
    import selective_state_space_160_b300 as msc
    from selective_state_space_160_b300.inputs import s6_inputs
    inp = s6_inputs(2, 32, 128, 16, seed=970, bf16=True)
    x, w, bias = _data(2, 32, 128, 4, 971, True)
    u = msc.msc_causal_conv1d_fwd(to_dev(x, True), to_dev(w), to_dev(bias), out_dtype=torch.bfloat16)
    dev = {k: to_dev(inp[k], True) for k in ("delta", "z", "B", "C")}
    y = msc.msc_selective_scan_fwd(u, dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], to_dev(inp["D"]),
                                   dev["z"], to_dev(inp["delta_bias"]))
    u_ref = _out_np(u)                       # the bf16 values the scan consumed
    assert bf16_match(u_ref, oracle.causal_conv1d(x, w, bias), x, w, bias) <= 1.0
    ref = oracle.s6_fwd(u_ref, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ref) <= 2e-3


def test_conv_config_full_size_sampled():
    """batch 8 x D 5120 x L 2048, K 4, bf16 in and out: the launch the bench
    times.  Channels 0, 1, 2047 and 5119 of every batch entry are checked."""
    import torch
    import selective_state_space_160_b300 as msc
    x, w, bias = _data(8, 5120, 2048, 4, 160_006, True)
    out = msc.msc_causal_conv1d_fwd(to_dev(x, True), to_dev(w), to_dev(bias), out_dtype=torch.bfloat16)
    got = _out_np(out)
    ds = [0, 1, 2047, 5119]
    ref = oracle.causal_conv1d(x[:, ds], w[ds], bias[ds])
    assert bf16_match(got[:, ds], ref, x[:, ds], w[ds], bias[ds]) <= 1.0
    assert np.all(np.isfinite(got))


# ----------------------------------------------------------------------------- backward
TOL_BWD = 1e-4


def _bwd(x, w, bias, dout, bf16, silu=True, with_dbias=True):
    import selective_state_space_160_b300 as msc
    dx, dw, db = msc.msc_causal_conv1d_bwd(to_dev(x, bf16), to_dev(w), to_dev(dout), to_dev(bias), silu=silu,
                                           with_dbias=with_dbias)
    return dx.cpu().numpy(), dw.cpu().numpy(), (None if db is None else db.cpu().numpy())


@pytest.mark.parametrize("batch,dim,L,K,bf16,silu", [
    (1, 4, 64, 4, False, True), (2, 37, 96, 4, True, True), (2, 5, 100, 3, False, True),
    (1, 3, 17, 8, False, False), (3, 8, 2048, 4, True, True), (1, 6, 1, 2, True, True),
    (2, 33, 999, 1, False, True), (2, 30, 1048, 4, False, True), (1, 5, 520, 3, True, False),
    (4, 700, 1024, 2, True, True)])
def test_bwd_shapes(batch, dim, L, K, bf16, silu):
    x, w, bias = _data(batch, dim, L, K, 5000 + L + K, bf16)
    dout = np.random.default_rng(5100 + L).standard_normal((batch, dim, L)).astype(np.float32)
    dx, dw, db = _bwd(x, w, bias, dout, bf16, silu)
    rdx, rdw, rdb = oracle.causal_conv1d_bwd(x, w, bias, dout, silu=silu)
    assert max_rel_err(dx, rdx) <= TOL_BWD
    # dw and db sum batch x L terms: relative to the sum of their magnitudes
    scale = 1.0 + np.abs(dout).sum() / dim
    assert np.max(np.abs(dw - rdw)) / scale <= TOL_BWD
    assert np.max(np.abs(db - rdb)) / scale <= TOL_BWD


def test_bwd_no_bias_and_no_dbias():
    x, w, _ = _data(2, 16, 256, 4, 5200, False)
    dout = np.random.default_rng(5201).standard_normal((2, 16, 256)).astype(np.float32)
    dx, dw, db = _bwd(x, w, None, dout, False, with_dbias=False)
    rdx, rdw, _ = oracle.causal_conv1d_bwd(x, w, None, dout)
    assert db is None
    assert max_rel_err(dx, rdx) <= TOL_BWD
    assert max_rel_err(dw, rdw) <= 1e-3


def test_bwd_through_scan_chain():
    """conv -> scan -> loss: the scan's du fed to the conv backward equals the
    oracle's chain (conv oracle, S6 backward oracle, conv backward oracle)."""
    import selective_state_space_160_b300 as msc
    from selective_state_space_160_b300.inputs import s6_inputs, conv_taps
    inp = s6_inputs(2, 24, 128, 16, seed=5300, with_dy=True)
    w, cb = conv_taps(24, 4, seed=5301)
    u = msc.msc_causal_conv1d_fwd(to_dev(inp["u"]), to_dev(w), to_dev(cb))
    g = msc.msc_selective_scan_bwd(u, to_dev(inp["delta"]), to_dev(inp["A"]), to_dev(inp["B"]), to_dev(inp["C"]),
                                   to_dev(inp["D"]), to_dev(inp["z"]), to_dev(inp["delta_bias"]), to_dev(inp["dy"]))
    dx, dw, db = msc.msc_causal_conv1d_bwd(to_dev(inp["u"]), to_dev(w), g["du"], to_dev(cb))
    ru = oracle.causal_conv1d(inp["u"], w, cb)
    rg = oracle.s6_bwd(ru, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"],
                       inp["dy"])
    rdx, rdw, rdb = oracle.causal_conv1d_bwd(inp["u"], w, cb, rg["du"])
    assert max_rel_err(dx.cpu().numpy(), rdx) <= 1e-3
    assert max_rel_err(dw.cpu().numpy(), rdw) <= 1e-3
    assert max_rel_err(db.cpu().numpy(), rdb) <= 1e-3


def test_bwd_config_full_size_sampled():
    """batch 8 x D 5120 x L 2048, K 4, bf16 x, fp32 dout: the launch the bench
    times.  dx, dweight and dbias of channels 0, 1, 2047 and 5119 (every batch
    entry and step) against the oracle on those channels."""
    x, w, bias = _data(8, 5120, 2048, 4, 160_010, True)
    dout = np.random.default_rng(160_011).standard_normal((8, 5120, 2048)).astype(np.float32)
    dx, dw, db = _bwd(x, w, bias, dout, True)
    assert np.all(np.isfinite(dx))
    ds = [0, 1, 2047, 5119]
    rdx, rdw, rdb = oracle.causal_conv1d_bwd(x[:, ds], w[ds], bias[ds], dout[:, ds])
    assert max_rel_err(dx[:, ds], rdx) <= TOL_BWD
    scale = 1.0 + np.abs(dout[:, ds]).sum() / len(ds)
    assert np.max(np.abs(dw[ds] - rdw)) / scale <= TOL_BWD
    assert np.max(np.abs(db[ds] - rdb)) / scale <= TOL_BWD
