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


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    import selective_state_space_160_b300 as msc
    lib = msc.load_library()
    # Few rows and a long sequence make the plan split rows into independent
    # segments, whose scratch (rows x segments x (dstate + 1) x 4 B) is required;
    # find such a shape on this GPU whose scratch exceeds the array (at these
    # channel counts the optional chained scratch is at most about 1 MB, so a
    # larger query is the required segment scratch).
    shape = None
    for dim in (4096, 8192, 16384):
        for L in (1 << 17, 1 << 19, 1 << 21):
            if msc.msc_selective_scan_fwd_workspace_size(1, dim, L, 16) > (4 << 20):
                shape = (dim, L)
                break
        if shape:
            break
    assert shape is not None
    dim, L = shape
    # The call is refused on the host before anything is launched, so small
    # device buffers stand in for the (multi-GB) inputs.
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    f = lib.msc_selective_scan_fwd_noalloc
    st = f(1, dim, L, 16, 0, p, p, p, p, p, None, None, None, None, p, None, None)
    assert st == msc.MSC_ERR_WORKSPACE
    assert "scratch" in msc.msc_last_error()
