"""The allocation-free S6 forward (msc_selective_scan_fwd_noalloc), for callers
that cannot allocate device memory (a plugin inside a framework that owns all
device allocations, or a serving loop that must not call cudaMalloc on its hot
path).  It is called through the C ABI and must match the workspace-taking
forward, twice in a row (the library-owned scratch keeps the previous call's
contents).  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from selective_state_space_160_b300.inputs import s6_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, dev, batch, dim, L, N, y, h_last, bf16):
    import torch
    f = lib.msc_selective_scan_fwd_noalloc
    ptr = lambda t: None if t is None else t.data_ptr()
    return f(batch, dim, L, N, 1 if bf16 else 0, ptr(dev["u"]), ptr(dev["delta"]), ptr(dev["A"]), ptr(dev["B"]),
             ptr(dev["C"]), ptr(dev["D"]), ptr(dev["z"]), ptr(dev["delta_bias"]), None, ptr(y), ptr(h_last),
             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("batch,dim,L,bf16", [(2, 64, 32768, False), (1, 3, 12345, True), (4, 256, 2048, True)])
def test_noalloc_matches_workspace_forward_twice(batch, dim, L, bf16):
    import torch
    import selective_state_space_160_b300 as msc
    lib = msc.load_library()
    N = 16
    inp = s6_inputs(batch, dim, L, N, seed=77 + L, bf16=bf16)
    dev = {k: to_dev(inp[k], bf16 and k in ("u", "delta", "z", "B", "C")) for k in
           ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")}
    ref_y, ref_h = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                              dev["z"], dev["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    for it in range(2):
        y = torch.full((batch, dim, L), float("nan"), dtype=torch.float32, device="cuda")
        h_last = torch.full((batch, dim, N), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        st = _call_noalloc(lib, dev, batch, dim, L, N, y, h_last, bf16)
        torch.cuda.synchronize()
        assert st == 0, msc.msc_last_error()
        if it == 1:
            # the second call on this device allocates no device memory at all
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_allocated() == alloc0
        msc.msc_check_device_status()
        tol = 2e-3 if bf16 else 1e-4
        assert max_rel_err(y.cpu().numpy(), ref_y.cpu().numpy()) <= tol
        assert max_rel_err(h_last.cpu().numpy(), ref_h.cpu().numpy()) <= tol


def test_noalloc_long_sequence_plans_within_its_scratch():
    """Few rows and a long sequence: the workspace forward would split the rows
    into more segments than the library's array can hold scratch for; the
    allocation-free call plans fewer segments and still matches it."""
    import torch
    import selective_state_space_160_b300 as msc
    lib = msc.load_library()
    batch, dim, L, N = 1, 4096, 1 << 16, 16
    assert msc.msc_selective_scan_fwd_workspace_size(batch, dim, L, N) > (4 << 20)
    g = torch.Generator(device="cuda").manual_seed(77)
    bf = torch.bfloat16
    dev = {"u": torch.randn((batch, dim, L), device="cuda", generator=g).to(bf),
           "delta": (0.5 * torch.randn((batch, dim, L), device="cuda", generator=g)).to(bf),
           "z": torch.randn((batch, dim, L), device="cuda", generator=g).to(bf),
           "B": torch.randn((batch, N, L), device="cuda", generator=g).to(bf),
           "C": torch.randn((batch, N, L), device="cuda", generator=g).to(bf),
           "A": -torch.arange(1, N + 1, device="cuda", dtype=torch.float32).repeat(dim, 1).contiguous(),
           "D": torch.ones(dim, device="cuda")}
    dt = torch.exp(torch.empty(dim, device="cuda").uniform_(np.log(1e-3), np.log(1e-1), generator=g))
    dev["delta_bias"] = torch.log(torch.expm1(dt))
    ref_y, ref_h = msc.msc_selective_scan_fwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                              dev["z"], dev["delta_bias"], return_last_state=True)
    y = torch.full_like(ref_y, float("nan"))
    h_last = torch.full_like(ref_h, float("nan"))
    torch.cuda.synchronize()
    assert _call_noalloc(lib, dev, batch, dim, L, N, y, h_last, True) == 0, msc.msc_last_error()
    torch.cuda.synchronize()
    msc.msc_check_device_status()
    # the two plans combine segments differently: fp32 rounding apart, the same values
    err = ((y - ref_y).abs() / (1 + ref_y.abs())).max().item()
    assert err <= 2e-3, err
    errh = ((h_last - ref_h).abs() / (1 + ref_h.abs())).max().item()
    assert errh <= 2e-3, errh
