"""GPU parity of the Mamba-2 SSD chunked backward (through the C ABI) against
the oracle's SSD backward, which composes the S6 backward over the channels
that share Delta, A (a head) and B, C (a group), and is pinned by finite
differences of the SSD forward.

bf16 inputs; tolerance max |gpu - ref| / (1 + |ref|) <= 2e-3 for every gradient."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import ssd_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-3
KEYS = ("dx", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def _run(inp, chunk, dy=None):
    import selective_state_space_160_b300 as msc
    dev = {k: to_dev(inp[k], True) for k in ("x", "delta", "B", "C", "z")}
    g = msc.msc_ssd_chunked_bwd(dev["x"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
                                to_dev(inp["dy"] if dy is None else dy, True), to_dev(inp["D"]), dev["z"],
                                to_dev(inp["delta_bias"]), chunk=chunk)
    return {k: v.cpu().numpy() for k, v in g.items()}


def _ref(inp, dy=None):
    return oracle.ssd_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                          inp["delta_bias"], inp["dy"] if dy is None else dy)


def _check(g, r, tol=TOL):
    for k in KEYS:
        if r.get(k) is None:
            assert g.get(k) is None, k
            continue
        e = max_rel_err(g[k], r[k])
        assert e <= tol, (k, e)


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("L", [256, 300])
def test_chunk_sizes_and_ragged_lengths(chunk, L):
    inp = ssd_inputs(1, L, 2, 64, 128, 1, seed=3000 + L + chunk, bf16=True, with_dy=True)
    _check(_run(inp, chunk), _ref(inp))


@pytest.mark.parametrize("with_z,with_D,with_bias", [(True, True, True), (True, False, True),
                                                     (False, True, False), (False, False, False)])
def test_optional_inputs(with_z, with_D, with_bias):
    inp = ssd_inputs(2, 520, 3, 64, 128, 1, seed=3100 + 4 * with_z + 2 * with_D + with_bias, bf16=True,
                     with_z=with_z, with_D=with_D, with_bias=with_bias, with_dy=True)
    _check(_run(inp, 256), _ref(inp))


def test_many_heads_and_groups():
    # 32 heads in 2 groups: dG, dB, dC summed over 16 heads per group
    inp = ssd_inputs(1, 384, 32, 64, 128, 2, seed=3200, bf16=True, with_dy=True, with_z=True)
    _check(_run(inp, 128), _ref(inp))
    # 20 heads, 1 group: a full and a partial block of 16 heads in the dB, dC state terms
    inp = ssd_inputs(2, 300, 20, 64, 128, 1, seed=3201, bf16=True, with_dy=True)
    _check(_run(inp, 256), _ref(inp))


def test_single_step_and_short():
    inp = ssd_inputs(1, 1, 2, 64, 128, 1, seed=3300, bf16=True, with_dy=True, with_z=True)
    _check(_run(inp, 64), _ref(inp))
    inp = ssd_inputs(1, 17, 2, 64, 128, 1, seed=3301, bf16=True, with_dy=True)
    _check(_run(inp, 256), _ref(inp))


def test_chunk_size_does_not_change_result():
    inp = ssd_inputs(1, 768, 4, 64, 128, 1, seed=3400, bf16=True, with_dy=True)
    g64, g256 = _run(inp, 64), _run(inp, 256)
    for k in g64:
        assert max_rel_err(g64[k], g256[k]) <= TOL, k


def test_repeat_calls_close():
    """Sums use fp32 atomics, so repeats agree to rounding; dx and dz have none."""
    inp = ssd_inputs(1, 512, 4, 64, 128, 1, seed=3500, bf16=True, with_dy=True, with_z=True)
    g1, g2 = _run(inp, 256), _run(inp, 256)
    for k in g1:
        assert max_rel_err(g1[k], g2[k]) <= 1e-5, k
    for k in ("dx", "dz"):
        assert np.array_equal(g1[k], g2[k]), k


def test_zero_upstream_gradient():
    inp = ssd_inputs(1, 200, 2, 64, 128, 1, seed=3600, bf16=True, with_dy=True, with_z=True)
    g = _run(inp, 128, dy=np.zeros_like(inp["dy"]))
    for k, v in g.items():
        assert np.all(v == 0), k


def test_ssd_config_full_size_sampled_heads():
    """batch 4, 80 heads, P 64, N 128, 1 group, L 4096, chunk 256, bf16, the
    full-size launch.  dy is kept on three sampled heads and zeroed elsewhere, so
    every gradient (dB, dC included) equals the oracle's on the three-head
    sub-problem, and the other heads' per-head gradients are exactly zero.  A
    second launch with the full dy gives the sampled heads' dx and dz bit for
    bit (they depend on no other head)."""
    inp = ssd_inputs(4, 4096, 80, 64, 128, 1, seed=160_005, bf16=True, with_dy=True, with_z=True)
    hs = np.array([0, 41, 79])
    dym = np.zeros_like(inp["dy"])
    dym[:, :, hs, :] = inp["dy"][:, :, hs, :]
    g = _run(inp, 256, dy=dym)
    sub = dict(inp)
    for k in ("x", "z", "dy"):
        sub[k] = inp[k][:, :, hs, :]
    sub["delta"] = inp["delta"][:, :, hs]
    for k in ("A", "D", "delta_bias"):
        sub[k] = inp[k][hs]
    r = _ref(sub)
    gs = dict(g)
    for k in ("dx", "dz"):
        gs[k] = g[k][:, :, hs, :]
    gs["ddelta"] = g["ddelta"][:, :, hs]
    for k in ("dA", "dD", "ddelta_bias"):
        gs[k] = g[k][hs]
    _check(gs, r)
    others = np.setdiff1d(np.arange(80), hs)
    assert np.all(g["dx"][:, :, others, :] == 0) and np.all(g["ddelta"][:, :, others] == 0)
    assert np.all(g["dA"][others] == 0)
    full = _run(inp, 256)
    assert all(np.all(np.isfinite(v)) for v in full.values())
    for k in ("dx", "dz"):
        assert np.array_equal(full[k][:, :, hs, :], g[k][:, :, hs, :]), k


def test_gated_backward_first_in_a_fresh_process():
    """The gated backward as the first SSD call of a process (it takes a path
    that no earlier call has configured), checked against the oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = """
import sys
sys.path.insert(0, %r); sys.path.insert(0, %r)
import numpy as np
from oracle import oracle
from selective_state_space_160_b300.inputs import ssd_inputs
from helpers import max_rel_err, to_dev
import selective_state_space_160_b300 as msc
inp = ssd_inputs(1, 300, 2, 64, 128, 1, seed=3700, bf16=True, with_z=True, with_dy=True)
dev = {k: to_dev(inp[k], True) for k in ("x", "delta", "B", "C", "z", "dy")}
g = msc.msc_ssd_chunked_bwd(dev["x"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], dev["dy"],
                            to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]), chunk=128)
r = oracle.ssd_bwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                   inp["delta_bias"], inp["dy"])
e = max(max_rel_err(v.cpu().numpy(), r[k]) for k, v in g.items())
print("ERR", e)
sys.exit(0 if e <= 2e-3 else 1)
""" % (root, os.path.join(root, "tests"))
    res = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-2000:]
