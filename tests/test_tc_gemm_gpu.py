"""The tcgen05 building block (shared-memory descriptors, instruction descriptor,
TMEM accumulate and load) that the SSD kernels are built on: one-CTA GEMMs
D = A B^T against a host matmul, with tiles written by CUDA cores and by TMA."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _lib():
    from selective_state_space_160_b300 import build as b
    lib = ctypes.CDLL(b.build_fixtures())
    lib.msc_probe_tc_gemm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.msc_probe_tc_gemm.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("use_tma", [0, 1])
@pytest.mark.parametrize("K,N", [(64, 64), (128, 128), (128, 256), (64, 16)])
def test_tc_gemm(bf16, use_tma, K, N):
    import torch
    g = torch.Generator().manual_seed(K * 1000 + N + use_tma)
    dt = torch.bfloat16 if bf16 else torch.float16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    ref = A.double() @ B.double().T
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.empty(128, N, dtype=torch.float32, device="cuda")
    rc = _lib().msc_probe_tc_gemm(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), K, N, int(bf16), use_tma, 0, 0)
    assert rc == 0, rc
    err = (D.double().cpu() - ref).abs().max().item() / (1 + ref.abs().max().item())
    assert err < 1e-5, err


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("a_mn,b_mn", [(1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("K,N", [(64, 64), (128, 128), (128, 256), (64, 192)])
def test_tc_gemm_mn_major(bf16, a_mn, b_mn, K, N):
    """Operands given transposed (M or N contiguous) and used MN-major."""
    import torch
    g = torch.Generator().manual_seed(K * 1000 + N + 7 * a_mn + b_mn)
    dt = torch.bfloat16 if bf16 else torch.float16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    ref = A.double() @ B.double().T
    Ad = (A.T.contiguous() if a_mn else A).cuda()
    Bd = (B.T.contiguous() if b_mn else B).cuda()
    D = torch.empty(128, N, dtype=torch.float32, device="cuda")
    rc = _lib().msc_probe_tc_gemm(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), K, N, int(bf16), 1, a_mn, b_mn)
    assert rc == 0, rc
    err = (D.double().cpu() - ref).abs().max().item() / (1 + ref.abs().max().item())
    assert err < 1e-5, err
