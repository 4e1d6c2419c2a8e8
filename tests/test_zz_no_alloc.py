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
    for _ in range(2):
        y = torch.full((batch, dim, L), float("nan"), dtype=torch.float32, device="cuda")
        h_last = torch.full((batch, dim, N), float("nan"), dtype=torch.float32, device="cuda")
        st = _call_noalloc(lib, dev, batch, dim, L, N, y, h_last, bf16)
        assert st == 0, msc.msc_last_error()
        msc.msc_check_device_status()
        tol = 2e-3 if bf16 else 1e-4
        assert max_rel_err(y.cpu().numpy(), ref_y.cpu().numpy()) <= tol
        assert max_rel_err(h_last.cpu().numpy(), ref_h.cpu().numpy()) <= tol


def test_noalloc_rejects_problems_beyond_its_scratch():
    import selective_state_space_160_b300 as msc
    lib = msc.load_library()
    # 37000 channels x 2048 steps need two segments per row: ~5 MB of scratch
    need = msc.msc_selective_scan_fwd_workspace_size(1, 37000, 2048, 16)
    assert need > (4 << 20)
    f = lib.msc_selective_scan_fwd_noalloc
    st = f(1, 37000, 2048, 16, 0, 256, 256, 256, 256, 256, None, None, None, None, 256, None, None)
    assert st == msc.MSC_ERR_WORKSPACE
    assert "scratch" in msc.msc_last_error()
