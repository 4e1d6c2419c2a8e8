"""GPU parity of the Mamba-2 SSD chunked forward (through the C ABI) against the
oracle's scalar-A recurrence (pinned to the materialised semiseparable form).
bf16 inputs; tolerance max |gpu - ref| / (1 + |ref|) <= 2e-3."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import ssd_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _run(inp, chunk, final=False):
    import selective_state_space_160_b300 as msc
    dev = {k: to_dev(inp[k], True) for k in ("x", "delta", "B", "C", "z")}
    out = msc.msc_ssd_chunked_fwd(dev["x"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"],
                                  to_dev(inp["D"]), dev["z"], to_dev(inp["delta_bias"]), chunk=chunk,
                                  return_final_state=final)
    if final:
        return out[0].cpu().numpy(), out[1].cpu().numpy()
    return out.cpu().numpy()


def _ref(inp, final=False):
    return oracle.ssd_fwd(inp["x"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                          inp["delta_bias"], return_final_state=final)


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("L", [256, 300, 1000])
def test_chunk_sizes_and_ragged_lengths(chunk, L):
    inp = ssd_inputs(1, L, 2, 64, 128, 1, seed=L + chunk, bf16=True)
    y, fs = _run(inp, chunk, final=True)
    ry, rfs = _ref(inp, final=True)
    assert max_rel_err(y, ry) <= TOL
    assert max_rel_err(fs, rfs) <= TOL


def test_gate_and_optional_inputs():
    inp = ssd_inputs(2, 520, 3, 64, 128, 1, seed=5, bf16=True, with_z=True, with_D=False, with_bias=True)
    assert max_rel_err(_run(inp, 256), _ref(inp)) <= TOL
    inp = ssd_inputs(1, 384, 2, 64, 128, 1, seed=6, bf16=True, with_z=False, with_D=True, with_bias=False)
    assert max_rel_err(_run(inp, 128), _ref(inp)) <= TOL


def test_many_heads_and_groups():
    # 32 heads in 2 groups: two head blocks of the kernels, B/C per group
    inp = ssd_inputs(1, 512, 32, 64, 128, 2, seed=8, bf16=True)
    assert max_rel_err(_run(inp, 256), _ref(inp)) <= TOL
    # 20 heads, 1 group: a partial head block
    inp = ssd_inputs(2, 300, 20, 64, 128, 1, seed=9, bf16=True)
    assert max_rel_err(_run(inp, 256), _ref(inp)) <= TOL


def test_single_step_and_short():
    inp = ssd_inputs(1, 1, 2, 64, 128, 1, seed=10, bf16=True)
    assert max_rel_err(_run(inp, 64), _ref(inp)) <= TOL
    inp = ssd_inputs(1, 17, 2, 64, 128, 1, seed=11, bf16=True, with_z=True)
    assert max_rel_err(_run(inp, 256), _ref(inp)) <= TOL


def test_chunk_size_does_not_change_result():
    inp = ssd_inputs(1, 768, 4, 64, 128, 1, seed=12, bf16=True)
    y64, y256 = _run(inp, 64), _run(inp, 256)
    assert max_rel_err(y64, y256) <= TOL


def test_ssd_config_full_size_sampled_heads():
    """batch 4, 80 heads, P 64, N 128, 1 group, L 4096, chunk 256, bf16,
    full-size launch; oracle on sampled heads (all batch entries, all steps)."""
    import selective_state_space_160_b300 as msc
    inp = ssd_inputs(4, 4096, 80, 64, 128, 1, seed=160_004, bf16=True)
    y, fs = _run(inp, 256, final=True)
    assert np.all(np.isfinite(y))
    hs = np.array([0, 17, 79])
    sub = dict(inp)
    sub["x"] = inp["x"][:, :, hs, :]
    sub["delta"] = inp["delta"][:, :, hs]
    sub["A"], sub["D"], sub["delta_bias"] = inp["A"][hs], inp["D"][hs], inp["delta_bias"][hs]
    ry, rfs = _ref(sub, final=True)
    assert max_rel_err(y[:, :, hs, :], ry) <= TOL
    assert max_rel_err(fs[:, hs], rfs) <= TOL
    msc.msc_check_device_status()


def test_large_cumulative_decay_near_the_diagonal():
    """A = -16 and Delta near 4: the in-chunk cumulative sum cs reaches about
    -16 000 by the end of a 256-step chunk, while the decays that matter (the
    diagonal and its neighbours, exp(cs_i - cs_j) for j close to i) are near 1
    ("Mamba 解密" sec. 6.2: M_ij = a_{j+1} ... a_i).  The kernel forms the
    exponent from the difference cs_i - cs_j, which is exact for nearby steps;
    forming cs_i log2(e) and cs_j log2(e) apart would round each to about 1e-3
    at this size.  The result must match the oracle to 5e-4, a quarter of the
    bf16 tolerance."""
    inp = ssd_inputs(1, 512, 16, 64, 128, seed=4242, with_z=True)
    inp["A"] = np.full_like(inp["A"], -16.0)
    inp["delta_bias"] = np.full_like(inp["delta_bias"], np.log(np.expm1(4.0)))
    y = _run(inp, 256)
    ref = _ref(inp)
    assert np.all(np.isfinite(y))
    assert max_rel_err(y, ref) <= 5e-4
