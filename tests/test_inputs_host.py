"""The seeded input recipe (CPU): the same seed gives the same arrays, the draws
follow the stated distributions and parameter initialisation, and bf16
rounding is round-to-nearest-even as torch's own conversion does it."""
import numpy as np
import pytest

from selective_state_space_160_b300.inputs import bf16_bits, bf16_round, conv_taps, s6_inputs, ssd_inputs


def _same(a, b):
    return all((a[k] is None and b[k] is None) or np.array_equal(a[k], b[k]) for k in a)


def test_seeded_and_reproducible():
    a = s6_inputs(2, 8, 64, 16, seed=5, with_dy=True)
    b = s6_inputs(2, 8, 64, 16, seed=5, with_dy=True)
    c = s6_inputs(2, 8, 64, 16, seed=6, with_dy=True)
    assert _same(a, b)
    assert not np.array_equal(a["u"], c["u"])
    s1 = ssd_inputs(1, 32, 4, 8, 16, ngroups=2, seed=9, with_z=True, with_dy=True)
    s2 = ssd_inputs(1, 32, 4, 8, 16, ngroups=2, seed=9, with_z=True, with_dy=True)
    assert _same(s1, s2)


def test_s6_distributions_and_parameters():
    inp = s6_inputs(4, 64, 1024, 16, seed=160_000, with_dy=True)
    for k, scale in (("u", 1.0), ("z", 1.0), ("B", 1.0), ("C", 1.0), ("dy", 1.0), ("delta", 0.5)):
        v = inp[k].astype(np.float64)
        assert abs(v.mean()) < 0.01 * scale, k
        assert abs(v.std() - scale) < 0.01 * scale, k
    # Delta_bias is the inverse softplus of dt ~ log-uniform[1e-3, 1e-1]
    dt = np.log1p(np.exp(inp["delta_bias"].astype(np.float64)))
    assert np.all(dt >= 1e-3 * (1 - 1e-5)) and np.all(dt <= 1e-1 * (1 + 1e-5))
    assert np.log(dt).min() < np.log(3e-3) and np.log(dt).max() > np.log(3e-2)   # spread over the range
    assert np.array_equal(inp["A"], np.tile(-np.arange(1, 17, dtype=np.float32), (64, 1)))
    assert np.array_equal(inp["D"], np.ones(64, np.float32))


def test_ssd_parameters():
    inp = ssd_inputs(1, 16, 80, 8, 16, seed=160_004)
    assert inp["A"].shape == (80,) and np.all(inp["A"] <= -1.0) and np.all(inp["A"] >= -16.0)
    assert inp["A"].min() < -12.0 and inp["A"].max() > -5.0
    dt = np.log1p(np.exp(inp["delta_bias"].astype(np.float64)))
    assert np.all((dt >= 1e-3 * (1 - 1e-5)) & (dt <= 1e-1 * (1 + 1e-5)))
    assert inp["z"] is None and np.array_equal(inp["D"], np.ones(80, np.float32))


def test_optional_inputs_absent():
    inp = s6_inputs(1, 4, 8, 4, with_z=False, with_D=False, with_bias=False)
    assert inp["z"] is None and inp["D"] is None and inp["delta_bias"] is None


def test_bf16_round_matches_torch_and_ties_to_even():
    import torch
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100_000), rng.standard_normal(1000) * 1e30,
                        rng.standard_normal(1000) * 1e-30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bf16_round(x), ref)
    # exactly halfway cases round to the even neighbour
    one = np.float32(1.0)
    half_ulp = np.float32(2.0 ** -8)
    assert bf16_round(np.array([one + half_ulp], np.float32))[0] == one                    # 1 is even
    odd = np.float32(1.0 + 2.0 ** -7)
    assert bf16_round(np.array([odd + half_ulp], np.float32))[0] == np.float32(1.0 + 2.0 ** -6)
    assert np.isnan(bf16_round(np.array([np.nan], np.float32))[0])
    # bf16 values are fixed points, and their bit patterns round-trip
    v = bf16_round(x)
    assert np.array_equal(bf16_round(v), v)
    bits = bf16_bits(v)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), v)


def test_conv_taps_scale():
    w, b = conv_taps(4096, 4, seed=1)
    assert w.shape == (4096, 4) and b.shape == (4096,)
    assert abs((w.astype(np.float64) ** 2).sum(axis=1).mean() - 1.0) < 0.05   # unit output variance
    assert abs(b.std() - 0.1) < 0.01


@pytest.mark.parametrize("bf16", [False, True])
def test_bf16_flag_rounds_streamed_inputs_only(bf16):
    inp = s6_inputs(1, 8, 32, 16, seed=11, bf16=bf16)
    for k in ("u", "delta", "z", "B", "C"):
        assert np.array_equal(bf16_round(inp[k]), inp[k]) or not bf16, k
    # parameters stay fp32 whatever the streamed dtype
    raw = s6_inputs(1, 8, 32, 16, seed=11, bf16=False)
    assert np.array_equal(inp["delta_bias"], raw["delta_bias"]) and np.array_equal(inp["A"], raw["A"])
