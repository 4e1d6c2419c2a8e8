"""GPU tests of the S6 training pair: msc_selective_scan_fwd_train (the forward
that also keeps the state entering every 8-step group) and
msc_selective_scan_bwd_ckpt (the backward that starts from those states instead
of recomputing them; the pages only fix that the backward recomputes states
rather than storing them all, bqwf survey sec. 2.2).

- y equals msc_selective_scan_fwd's bit for bit, on every plan (one pass,
  chained chunks, segments);
- the checkpoints match the oracle's state after 8g steps on sampled rows;
- with the forward in one pass or in chained chunks, the gradients written
  without atomics (du, ddelta, dz) equal msc_selective_scan_bwd's bit for bit
  -- which holds only if the checkpoints are the ones the backward computes
  itself -- and the atomic sums agree to 1e-5; with segments (whose carries
  combine the states in another order) every gradient agrees to 1e-5;
- on a small case every gradient matches the oracle."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, s6_inputs_torch
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-3


def _args(inp):
    return (inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])


@pytest.mark.parametrize("batch,dim,L,bf16,bitwise", [
    (2, 37, 64, True, True),        # one pass, partial row block
    (1, 36, 48, False, True),       # fp32 16-step tiles
    (1, 24000, 1024, True, True),   # chained chunks on persistent CTAs
    (2, 33, 2048, True, False),     # few rows: 4 segments of 512 steps
    (1, 3, 5000, False, False),     # few rows, long: segments (aggregate, carry, full with checkpoints)
])
def test_pair_matches_plain_forward_and_backward(batch, dim, L, bf16, bitwise):
    import torch
    import selective_state_space_160_b300 as msc
    N = 16
    inp = s6_inputs_torch(batch, dim, L, N, seed=41_000 + dim + L, bf16=bf16)
    g = torch.Generator(device="cuda").manual_seed(21)
    dy = torch.randn((batch, dim, L), device="cuda", generator=g)
    dy = dy.to(torch.bfloat16) if bf16 else dy
    assert msc.msc_selective_scan_ckpt_size(batch, dim, L, N) == batch * dim * (L // 8) * 16 * 4
    y_plain = msc.msc_selective_scan_fwd(*_args(inp))
    y_train, ckpt = msc.msc_selective_scan_fwd_train(*_args(inp))
    torch.cuda.synchronize()
    assert bool(torch.equal(y_train, y_plain))
    g_plain = msc.msc_selective_scan_bwd(*_args(inp), dy)
    g_pair = msc.msc_selective_scan_bwd_ckpt(*_args(inp), dy, ckpt)
    torch.cuda.synchronize()
    msc.msc_check_device_status()
    # du does not depend on the states: equal on every plan
    assert bool(torch.equal(g_pair["du"], g_plain["du"]))
    for k in (("ddelta", "dz") if bitwise else ()):
        assert bool(torch.equal(g_pair[k], g_plain[k])), k
    for k in ("ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        a, b = g_pair[k].double(), g_plain[k].double()
        assert float((a - b).abs().max() / (1.0 + b.abs().max())) <= 1e-5, k
    # checkpoints against the oracle: the state entering group gi of a row is the
    # state after 8 gi steps from zero
    host = {k: inp[k].float().cpu().numpy() for k in ("B", "C")}
    ck = ckpt.view(batch * dim, L // 8, 16).cpu().numpy()
    for d in (0, dim - 1):
        for gi in (1, (L // 8) // 2, L // 8 - 1):
            t = 8 * gi
            sub = {k: inp[k][:1, d:d + 1, :t].float().cpu().numpy() for k in ("u", "delta", "z")}
            _, h = oracle.s6_fwd(sub["u"], sub["delta"], inp["A"][d:d + 1].cpu().numpy(), host["B"][:1, :, :t],
                                 host["C"][:1, :, :t], inp["D"][d:d + 1].cpu().numpy(), sub["z"],
                                 inp["delta_bias"][d:d + 1].cpu().numpy(), return_last_state=True)
            assert max_rel_err(ck[d, gi][None, None, :], h) <= TOL_BF16, (d, gi)
    del inp, y_plain, y_train, ckpt, g_plain, g_pair
    torch.cuda.empty_cache()


def test_pair_gradients_against_the_oracle():
    import selective_state_space_160_b300 as msc
    batch, dim, L, N = 2, 24, 64, 16
    inp = s6_inputs(batch, dim, L, N, seed=41_500, bf16=True, with_dy=True)
    dev = {k: to_dev(inp[k], True) for k in ("u", "delta", "z", "B", "C", "dy")}
    args = (dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], to_dev(inp["D"]), dev["z"],
            to_dev(inp["delta_bias"]))
    y, ckpt = msc.msc_selective_scan_fwd_train(*args)
    grads = msc.msc_selective_scan_bwd_ckpt(*args, dev["dy"], ckpt)
    ry = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                       inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ry) <= TOL_BF16
    ref = oracle.s6_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                        inp["delta_bias"], inp["dy"])
    for k, v in ref.items():
        if v is None or grads.get(k) is None:
            continue
        assert max_rel_err(grads[k].cpu().numpy(), v) <= TOL_BF16, k


def test_pair_limits():
    """seqlen not a multiple of 8, more than 16 states: refused before any
    launch; the checkpoint size query returns 0 for them."""
    import selective_state_space_160_b300 as msc
    assert msc.msc_selective_scan_ckpt_size(1, 4, 60, 16) == 0
    assert msc.msc_selective_scan_ckpt_size(1, 4, 64, 17) == 0
    inp = s6_inputs(1, 4, 60, 16, seed=41_600)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "z", "B", "C")}
    args = (d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]), d["z"],
            to_dev(inp["delta_bias"]))
    import torch
    with pytest.raises(msc.MscError) as e:
        msc.msc_selective_scan_fwd_train(*args, ckpt=torch.empty(64, device="cuda"))
    assert e.value.status == msc.MSC_ERR_UNSUPPORTED and "multiple of 8" in str(e.value)
    msc.msc_check_device_status()


@pytest.mark.parametrize("with_z,with_D,with_bias,bf16", [(False, True, True, True), (True, False, False, False),
                                                          (False, False, False, True)])
def test_pair_optional_inputs_against_the_oracle(with_z, with_D, with_bias, bf16):
    import selective_state_space_160_b300 as msc
    batch, dim, L, N = 2, 33, 96, 16
    inp = s6_inputs(batch, dim, L, N, seed=41_700 + 4 * with_z + 2 * with_D + with_bias, bf16=bf16, with_dy=True,
                    with_z=with_z, with_D=with_D, with_bias=with_bias)
    dev = {k: (to_dev(inp[k], bf16) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C", "dy")}
    args = (dev["u"], dev["delta"], to_dev(inp["A"]), dev["B"], dev["C"], to_dev(inp["D"]), dev["z"],
            to_dev(inp["delta_bias"]))
    y, ckpt = msc.msc_selective_scan_fwd_train(*args)
    grads = msc.msc_selective_scan_bwd_ckpt(*args, dev["dy"], ckpt)
    tol = TOL_BF16 if bf16 else 1e-3
    ry = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                       inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ry) <= (TOL_BF16 if bf16 else 1e-4)
    ref = oracle.s6_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                        inp["delta_bias"], inp["dy"])
    for k, v in ref.items():
        if v is None or grads.get(k) is None:
            assert grads.get(k) is None or v is None, k
            continue
        assert max_rel_err(grads[k].cpu().numpy(), v) <= tol, k
