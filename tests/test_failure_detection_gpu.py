"""Failure detection on the GPU without a fault: the library's bounded wait,
run on a barrier that nothing completes, gives up after about one second and
reports MSC_ERR_TIMEOUT; the context stays usable (a forward afterwards matches
the oracle and the device status words are clear)."""
import ctypes

import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu


def _probe():
    from selective_state_space_160_b300 import build as b
    lib = ctypes.CDLL(b.build_fixtures())
    lib.msc_probe_wait_timeout.restype = ctypes.c_int
    lib.msc_probe_wait_timeout.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint),
                                           ctypes.POINTER(ctypes.c_double)]
    return lib


def test_wait_that_nothing_completes_times_out_and_the_gpu_stays_usable():
    import selective_state_space_160_b300 as msc
    lib = _probe()
    st, secs = ctypes.c_uint(99), ctypes.c_double(-1.0)
    assert lib.msc_probe_wait_timeout(0, ctypes.byref(st), ctypes.byref(secs)) == 0
    assert st.value == msc.MSC_ERR_TIMEOUT
    assert 0.9 <= secs.value <= 5.0, secs.value
    # the same wait completes at once when the barrier is completed
    assert lib.msc_probe_wait_timeout(1, ctypes.byref(st), ctypes.byref(secs)) == 0
    assert st.value == 0 and secs.value < 0.1
    # the context is usable: a forward matches the oracle, status words clear
    inp = s6_inputs(1, 16, 96, 16, seed=8000, bf16=True)
    y = msc.msc_selective_scan_fwd(*(to_dev(inp[k], k in ("u", "delta", "B", "C", "z"))
                                     for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")))
    ref = oracle.s6_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                        inp["delta_bias"])
    assert max_rel_err(y.cpu().numpy(), ref) <= 2e-3
    msc.msc_check_device_status()   # raises if a status word is set
