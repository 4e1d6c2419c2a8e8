"""GPU parity of the S6 forward on rows of 2^19 steps or more, where the full
pass stages y in shared memory and writes each row's 32-step window as one
128-byte run (with bf16 inputs a window is one tile, with fp32 two; a row's
last window may be ragged or hold a single tile).  Every discretisation, the
fused conv front end, the initial and final state, few rows (segments) and a
second batch entry, each against the oracle on every row.

Tolerances (max |gpu - ref| / (1 + |ref|)): 1e-4 with fp32 inputs, 2e-3 with
bf16 inputs (the oracle consumes the same bf16-rounded values)."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, conv_taps
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

L0 = 1 << 19


@pytest.mark.parametrize("batch,dim,L,bf16,disc", [
    (1, 3, L0 + 24, True, oracle.DISC_EULER),       # last window 24 of 32 steps
    (1, 5, L0 + 20, False, oracle.DISC_ZOH),        # fp32: last window one ragged tile
    (2, 2, L0 + 8, True, oracle.DISC_TRAPEZOID),
    (1, 33, L0 + 48, False, oracle.DISC_EULER),     # a ragged second row block
])
def test_long_rows_against_the_oracle(batch, dim, L, bf16, disc):
    import selective_state_space_160_b300 as msc
    inp = s6_inputs(batch, dim, L, 16, seed=52_000 + dim + disc, bf16=bf16)
    h0 = np.random.default_rng(52_100 + dim).standard_normal((batch, dim, 16)).astype(np.float32)
    dev = {k: to_dev(inp[k], bf16) for k in ("u", "delta", "z", "B", "C")}
    y, hl = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
                                       to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]), h0=to_dev(h0),
                                       return_last_state=True, disc=disc)
    ry, rh = oracle.s6_fwd_disc(disc, inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], h0=h0, return_last_state=True)
    tol = 2e-3 if bf16 else 1e-4
    assert max_rel_err(y.cpu().numpy(), ry) <= tol
    assert max_rel_err(hl.cpu().numpy(), rh) <= tol


@pytest.mark.parametrize("bf16", [True, False])
def test_long_rows_fused_conv(bf16):
    import selective_state_space_160_b300 as msc
    batch, dim, L = 1, 4, L0 + 40
    inp = s6_inputs(batch, dim, L, 16, seed=52_200 + bf16, bf16=bf16)
    w, cb = conv_taps(dim, 4, seed=52_201)
    dev = {k: to_dev(inp[k], bf16) for k in ("u", "delta", "z", "B", "C")}
    y = msc.msc_selective_scan_fwd_conv(dev["u"], to_dev(w), to_dev(cb), dev["delta"], to_dev(inp["A"]), dev["B"],
                                        dev["C"], to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]))
    u = oracle.causal_conv1d(inp["u"], w, cb)
    ry = oracle.s6_fwd(u, inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ry) <= (2e-3 if bf16 else 1e-4)


def test_long_rows_without_gate_and_skip():
    """z, D and Delta_bias left out: the staged window holds C h alone."""
    import selective_state_space_160_b300 as msc
    batch, dim, L = 1, 2, L0 + 4
    inp = s6_inputs(batch, dim, L, 16, seed=52_300, with_z=False, with_D=False, with_bias=False)
    dev = {k: (to_dev(inp[k]) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C")}
    y = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], to_dev(inp["D"]),
                                   dev["z"], to_dev(inp["delta_bias"]))
    ry = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ry) <= 1e-4
