"""GPU parity of the S6 decode step (msc_selective_state_update, through the C
ABI) against the oracle's decode step, and against the scan run over the same
tokens, for 1 to 64 states (two, four or eight lanes per row).

Tolerances (max |gpu - ref| / (1 + |ref|)): 1e-4 with fp32 inputs, 2e-3 with
bf16 inputs (the oracle consumes the same bf16-rounded values); chained steps
accumulate one fp32 rounding per step, the same as the scan."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-3


def _steps(inp, bf16, h0, T):
    """Run T decode steps on the GPU; returns (y [b, dim, T], final state)."""
    import selective_state_space_160_b300 as msc
    import torch
    state = to_dev(h0).contiguous()
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    ys = []
    for t in range(T):
        col = lambda k: None if inp[k] is None else to_dev(np.ascontiguousarray(inp[k][:, :, t]), bf16)
        y = msc.msc_selective_state_update(col("u"), col("delta"), A, col("B"), col("C"), D, col("z"), bias,
                                           state=state)
        ys.append(y.cpu().numpy())
    torch.cuda.synchronize()
    return np.stack(ys, axis=2), state.cpu().numpy()


def _oracle_steps(inp, h0, T):
    h = h0
    ys = []
    for t in range(T):
        zt = None if inp["z"] is None else inp["z"][:, :, t]
        y, h = oracle.s6_step(inp["u"][:, :, t], inp["delta"][:, :, t], inp["A"], inp["B"][:, :, t],
                              inp["C"][:, :, t], inp["D"], zt, inp["delta_bias"], h)
        ys.append(y)
    return np.stack(ys, axis=2), h


@pytest.mark.parametrize("batch,dim,N", [(1, 4, 16), (3, 37, 16), (2, 130, 16), (1, 5, 7), (4, 33, 1),
                                         (2, 64, 12), (1, 1, 16),
                                         # four and eight lanes per row: vector and scalar state rows
                                         (2, 37, 32), (3, 9, 20), (2, 33, 64), (1, 70, 48), (1, 3, 17)])
@pytest.mark.parametrize("bf16", [False, True])
def test_single_step(batch, dim, N, bf16):
    inp = s6_inputs(batch, dim, 1, N, seed=7000 + batch * 100 + dim + N, bf16=bf16)
    h0 = np.random.default_rng(batch + dim).standard_normal((batch, dim, N)).astype(np.float32)
    y, h = _steps(inp, bf16, h0, 1)
    yr, hr = _oracle_steps(inp, h0, 1)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y, yr) <= tol
    assert max_rel_err(h, hr) <= tol


@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, True, True), (True, False, False),
                                                     (False, False, False)])
def test_optional_inputs(with_z, with_D, with_bias):
    inp = s6_inputs(2, 40, 3, 16, seed=71, with_z=with_z, with_D=with_D, with_bias=with_bias)
    h0 = np.zeros((2, 40, 16), np.float32)
    y, h = _steps(inp, False, h0, 3)
    yr, hr = _oracle_steps(inp, h0, 3)
    assert max_rel_err(y, yr) <= TOL_F32
    assert max_rel_err(h, hr) <= TOL_F32


@pytest.mark.parametrize("bf16,N", [(False, 16), (True, 16), (True, 64), (False, 40)])
def test_steps_match_scan(bf16, N):
    """64 decode steps from a random state equal the GPU scan over the same 64
    tokens from that state, and both match the oracle scan."""
    import selective_state_space_160_b300 as msc
    T = 64
    inp = s6_inputs(2, 96, T, N, seed=72 + N, bf16=bf16)
    h0 = np.random.default_rng(3).standard_normal((2, 96, N)).astype(np.float32)
    y_step, h_step = _steps(inp, bf16, h0, T)
    dev = {k: to_dev(inp[k], bf16) for k in ("u", "delta", "z", "B", "C")}
    y_scan, h_scan = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
                                                to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]),
                                                h0=to_dev(h0), return_last_state=True)
    yr, hr = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                           inp["delta_bias"], h0=h0, return_last_state=True)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y_step, yr) <= tol
    assert max_rel_err(h_step, hr) <= tol
    assert max_rel_err(y_step, y_scan.cpu().numpy()) <= tol
    assert max_rel_err(h_step, h_scan.cpu().numpy()) <= tol


def test_decode_config_full_size_sampled():
    """batch 64 x D 5120 x N 16, bf16 inputs: the launch the bench times.
    Every row of batch entries 0 and 63 is checked against the oracle."""
    inp = s6_inputs(64, 5120, 1, 16, seed=160_005, bf16=True)
    h0 = np.random.default_rng(11).standard_normal((64, 5120, 16)).astype(np.float32)
    y, h = _steps(inp, True, h0, 1)
    for bsel in (0, 63):
        sub = {k: (v[bsel:bsel + 1] if (v is not None and k in ("u", "delta", "z", "B", "C")) else v)
               for k, v in inp.items()}
        yr, hr = _oracle_steps(sub, h0[bsel:bsel + 1], 1)
        assert max_rel_err(y[bsel:bsel + 1], yr) <= TOL_BF16
        assert max_rel_err(h[bsel:bsel + 1], hr) <= TOL_BF16
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(h))
