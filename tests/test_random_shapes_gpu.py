"""Randomised parity sweep: seeded draws of shapes and options for the S6
forward (every discretisation, 1..64 states, optional inputs, initial state,
aligned and unaligned rows: the plain-load kernel, the padded copies), the S6 backward, the decode step and the SSD
forward, each checked against the oracle on the same inputs.  The draws are
fixed by the seed, so a failure names a reproducible case; sizes stay small
enough for the oracle to finish in seconds.

Tolerances (max |gpu - ref| / (1 + |ref|)): forward 1e-4 with fp32 inputs,
gradients 1e-3 with fp32 inputs, 2e-3 with bf16 inputs."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, ssd_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu


def _draw_fwd(i):
    r = np.random.default_rng(90_000 + i)
    bf16 = bool(r.integers(2))
    disc = int(r.integers(3))
    N = int(r.choice([1, 3, 8, 16, 16, 17, 24, 32, 40, 64]))
    L = int(r.choice([1, 7, 8, 33, 64, 100, 256, 520, 1031, 2048]))
    if disc == 2 and N > 16:
        # the trapezoid above 16 states takes only rows TMA streams as they are
        m = 8 if bf16 else 4
        L = max(m, (L // m) * m)
    dim = int(r.integers(1, 80))
    batch = int(r.integers(1, 4))
    opts = dict(with_z=bool(r.integers(2)), with_D=bool(r.integers(2)), with_bias=bool(r.integers(2)))
    use_h0 = bool(r.integers(2))
    return batch, dim, L, N, bf16, disc, opts, use_h0


@pytest.mark.parametrize("i", range(48))
def test_forward_random(i):
    import selective_state_space_160_b300 as msc
    batch, dim, L, N, bf16, disc, opts, use_h0 = _draw_fwd(i)
    inp = s6_inputs(batch, dim, L, N, seed=91_000 + i, bf16=bf16, **opts)
    h0 = np.random.default_rng(i).standard_normal((batch, dim, N)).astype(np.float32) if use_h0 else None
    d = {k: (to_dev(inp[k], bf16) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C")}
    y, hl = msc.msc_selective_scan_fwd(d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                       d["z"], to_dev(inp["delta_bias"]), h0=None if h0 is None else to_dev(h0),
                                       return_last_state=True, disc=disc)
    ry, rh = oracle.s6_fwd_disc(disc, inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], h0=h0, return_last_state=True)
    tol = 2e-3 if bf16 else 1e-4
    case = (batch, dim, L, N, bf16, disc, opts, use_h0)
    assert max_rel_err(y.cpu().numpy(), ry) <= tol, case
    assert max_rel_err(hl.cpu().numpy(), rh) <= tol, case


@pytest.mark.parametrize("i", range(16))
def test_backward_random(i):
    import selective_state_space_160_b300 as msc
    r = np.random.default_rng(92_000 + i)
    bf16 = bool(r.integers(2))
    N = int(r.choice([1, 4, 16, 16, 24, 40]))
    L = int(r.choice([1, 9, 48, 64, 130, 300]))
    dim, batch = int(r.integers(1, 40)), int(r.integers(1, 3))
    opts = dict(with_z=bool(r.integers(2)), with_D=bool(r.integers(2)), with_bias=bool(r.integers(2)))
    inp = s6_inputs(batch, dim, L, N, seed=93_000 + i, bf16=bf16, with_dy=True, **opts)
    d = {k: (to_dev(inp[k], bf16) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C", "dy")}
    g = msc.msc_selective_scan_bwd(d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                   d["z"], to_dev(inp["delta_bias"]), d["dy"])
    ref = oracle.s6_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                        inp["delta_bias"], inp["dy"])
    tol = 2e-3 if bf16 else 1e-3
    for k, v in ref.items():
        if v is None or g.get(k) is None:
            continue
        assert max_rel_err(g[k].cpu().numpy(), v) <= tol, (k, batch, dim, L, N, bf16, opts)


@pytest.mark.parametrize("i", range(10))
def test_decode_step_random(i):
    import selective_state_space_160_b300 as msc
    r = np.random.default_rng(94_000 + i)
    bf16 = bool(r.integers(2))
    N = int(r.choice([1, 5, 16, 24, 32, 64]))
    dim, batch = int(r.integers(1, 70)), int(r.integers(1, 5))
    inp = s6_inputs(batch, dim, 1, N, seed=95_000 + i, bf16=bf16)
    st0 = np.random.default_rng(i).standard_normal((batch, dim, N)).astype(np.float32)
    col = {k: np.ascontiguousarray(inp[k][:, :, 0]) for k in ("u", "delta", "z", "B", "C")}
    state = to_dev(st0)
    y = msc.msc_selective_state_update(to_dev(col["u"], bf16), to_dev(col["delta"], bf16), to_dev(inp["A"]),
                                       to_dev(col["B"], bf16), to_dev(col["C"], bf16), to_dev(inp["D"]),
                                       to_dev(col["z"], bf16), to_dev(inp["delta_bias"]), state=state)
    ry, rs = oracle.s6_step(col["u"], col["delta"], inp["A"], col["B"], col["C"], inp["D"], col["z"],
                            inp["delta_bias"], st0)
    tol = 2e-3 if bf16 else 1e-4
    assert max_rel_err(y.cpu().numpy(), ry) <= tol
    assert max_rel_err(state.cpu().numpy(), rs) <= tol


@pytest.mark.parametrize("i", range(10))
def test_ssd_forward_random(i):
    import selective_state_space_160_b300 as msc
    r = np.random.default_rng(96_000 + i)
    chunk = int(r.choice([64, 128, 256]))
    L = int(r.integers(1, 700))
    G = int(r.choice([1, 1, 2]))
    H = int(r.choice([1, 2, 3, 5])) if G == 1 else 32
    batch = int(r.integers(1, 3))
    opts = dict(with_z=bool(r.integers(2)), with_D=bool(r.integers(2)), with_bias=bool(r.integers(2)))
    inp = ssd_inputs(batch, L, H, 64, 128, G, seed=97_000 + i, bf16=True, **opts)
    d = {k: (to_dev(inp[k], True) if inp[k] is not None else None) for k in ("x", "delta", "B", "C", "z")}
    y, fs = msc.msc_ssd_chunked_fwd(d["x"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                    d["z"], to_dev(inp["delta_bias"]), chunk=chunk, return_final_state=True)
    ry, rf = oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                            inp["delta_bias"], return_final_state=True)
    case = (batch, L, H, G, chunk, opts)
    assert max_rel_err(y.cpu().numpy(), ry) <= 2e-3, case
    assert max_rel_err(fs.cpu().numpy(), rf) <= 2e-3, case
