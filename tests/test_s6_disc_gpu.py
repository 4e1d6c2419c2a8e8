"""GPU parity of the S6 forward with the zero-order-hold and exponential-
trapezoidal input terms (msc_selective_scan_fwd_ex, through the C ABI) against
the oracle's discretisation variants.

Tolerances (max |gpu - ref| / (1 + |ref|)): 1e-4 with fp32 inputs, 2e-3 with
bf16 inputs (the oracle consumes the same bf16-rounded values)."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-3
DISCS = [oracle.DISC_ZOH, oracle.DISC_TRAPEZOID]


def _run(inp, bf16, disc, h0=None):
    import selective_state_space_160_b300 as msc
    dev = {k: to_dev(inp[k], bf16) for k in ("u", "delta", "z", "B", "C")}
    y, hl = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
                                       to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]),
                                       h0=None if h0 is None else to_dev(h0), return_last_state=True, disc=disc)
    return y.cpu().numpy(), hl.cpu().numpy()


def _ref(inp, disc, h0=None):
    return oracle.s6_fwd_disc(disc, inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                              inp["delta_bias"], h0=h0, return_last_state=True)


def _check(got, ref, tol):
    assert max_rel_err(got[0], ref[0]) <= tol
    assert max_rel_err(got[1], ref[1]) <= tol


@pytest.mark.parametrize("disc", DISCS)
@pytest.mark.parametrize("batch,dim,L,N,bf16", [(1, 4, 64, 16, False), (2, 37, 96, 16, True), (3, 40, 1000, 16, True),
                                                (2, 33, 1004, 16, False), (1, 70, 256, 4, False), (2, 6, 8, 16, True),
                                                (1, 64, 8192, 16, True)])
def test_shapes(disc, batch, dim, L, N, bf16):
    """Ragged tails (1000 = 31 tiles + 8 steps, 1004 with fp32 tiles of 16), few
    states, a single group, and 1 x 64 x 8192, which the plan splits into
    segments chained by the carry pass."""
    inp = s6_inputs(batch, dim, L, N, seed=3000 + 7 * disc + batch + dim + L + N, bf16=bf16)
    _check(_run(inp, bf16, disc), _ref(inp, disc), TOL_BF16 if bf16 else TOL_F32)


@pytest.mark.parametrize("disc", DISCS)
@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, True, True), (True, False, False)])
def test_optional_inputs_and_h0(disc, with_z, with_D, with_bias):
    inp = s6_inputs(2, 36, 128, 16, seed=3100 + disc, with_z=with_z, with_D=with_D, with_bias=with_bias)
    h0 = np.random.default_rng(disc).standard_normal((2, 36, 16)).astype(np.float32)
    _check(_run(inp, False, disc, h0), _ref(inp, disc, h0), TOL_F32)


def test_euler_through_ex_is_the_plain_forward():
    import selective_state_space_160_b300 as msc
    inp = s6_inputs(2, 40, 256, 16, seed=3200, bf16=True)
    dev = {k: to_dev(inp[k], True) for k in ("u", "delta", "z", "B", "C")}
    args = (dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], to_dev(inp["D"]), dev["z"],
            to_dev(inp["delta_bias"]))
    y0 = msc.msc_selective_scan_fwd(*args).cpu().numpy()
    y1 = _run(inp, True, msc.MSC_DISC_EULER)[0]
    assert np.array_equal(y0, y1)


@pytest.mark.parametrize("disc", DISCS)
@pytest.mark.parametrize("batch,dim,L,bf16", [(1, 4, 63, True), (2, 37, 61, False), (1, 3, 4097, True)])
def test_unaligned_rows_through_the_plain_kernel(disc, batch, dim, L, bf16):
    """Rows whose byte stride is not a multiple of 16 take the plain-load kernel,
    which runs every form; L 4097 with few rows takes segments (the trapezoid's
    half-term from the step before each segment)."""
    inp = s6_inputs(batch, dim, L, 16, seed=3300 + L + disc, bf16=bf16)
    h0 = np.random.default_rng(L).standard_normal((batch, dim, 16)).astype(np.float32)
    _check(_run(inp, bf16, disc, h0=h0), _ref(inp, disc, h0=h0), 2e-3 if bf16 else 1e-4)


@pytest.mark.parametrize("disc", DISCS)
def test_plain_and_tma_kernels_agree(disc, monkeypatch):
    """Aligned rows sent to the plain-load kernel (MSC_S6_FWD_PLAIN) give the
    TMA kernel's results to 1e-5."""
    inp = s6_inputs(2, 40, 256, 16, seed=3400 + disc, bf16=True)
    y_tma, h_tma = _run(inp, True, disc)
    monkeypatch.setenv("MSC_S6_FWD_PLAIN", "1")
    y_plain, h_plain = _run(inp, True, disc)
    assert max_rel_err(y_plain, y_tma) <= 1e-5
    assert max_rel_err(h_plain, h_tma) <= 1e-5


@pytest.mark.parametrize("disc", DISCS)
def test_headline_config_sampled(disc):
    """batch 8, D 5120, L 2048, N 16, bf16: batch entry 0 channels 0, 1, 2560,
    5119 and batch entry 7 channel 4095 against the oracle."""
    inp = s6_inputs(8, 5120, 2048, 16, seed=160_001, bf16=True)
    y, hl = _run(inp, True, disc)
    for bsel, ds in ((0, [0, 1, 2560, 5119]), (7, [4095])):
        sub = {k: (v[bsel:bsel + 1, ds] if (v is not None and k in ("u", "delta", "z")) else v)
               for k, v in inp.items()}
        sub["B"], sub["C"] = inp["B"][bsel:bsel + 1], inp["C"][bsel:bsel + 1]
        sub["A"], sub["D"], sub["delta_bias"] = inp["A"][ds], inp["D"][ds], inp["delta_bias"][ds]
        ry, rh = _ref(sub, disc)
        assert max_rel_err(y[bsel:bsel + 1, ds], ry) <= TOL_BF16
        assert max_rel_err(hl[bsel:bsel + 1, ds], rh) <= TOL_BF16
