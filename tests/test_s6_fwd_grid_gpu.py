"""The chained forward sizes its persistent grid from an occupancy query that
must belong to the kernel instance being launched.  A process whose first
chained forward had 64 states (three resident CTAs per SM) then runs the
16-state headline forward (batch 8 x 5120 x 2048, bf16; eight per SM) as fast
as a fresh process does: a cache shared by all instances would launch the
16-state forward on the 64-state grid, at about half the speed."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

SCRIPT = """
import sys, statistics
sys.path.insert(0, %r)
import torch
import selective_state_space_160_b300 as msc
from selective_state_space_160_b300.inputs import s6_inputs_torch

def run(inp, reps):
    b, d, L = inp["u"].shape
    N = inp["A"].shape[1]
    ws = torch.empty(msc.msc_selective_scan_fwd_workspace_size(b, d, L, N) + 1024, dtype=torch.uint8, device="cuda")
    y = torch.empty((b, d, L), dtype=torch.float32, device="cuda")
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        msc.msc_selective_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                   inp["delta_bias"], y=y, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    msc.msc_check_device_status()
    return statistics.median(times[3:])

if %r:
    run(s6_inputs_torch(8, 5120, 512, 64, seed=77, bf16=True), 4)   # chained, 64 state slots
print("MS", run(s6_inputs_torch(8, 5120, 2048, 16, seed=78, bf16=True), 13))
"""


def _time(wide_first):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", SCRIPT % (root, wide_first)], capture_output=True, text=True,
                         timeout=900)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-2000:]
    return float([l for l in res.stdout.splitlines() if l.startswith("MS ")][-1].split()[1])


def test_headline_grid_does_not_depend_on_the_first_instance():
    # one re-measurement of both before failing, so that a passing slowdown of a
    # shared GPU is not taken for the grid (the fault it guards against costs
    # a third: 0.582 against 0.436 ms)
    for attempt in range(2):
        fresh = _time(False)
        after_wide = _time(True)
        if after_wide <= 1.25 * fresh:
            break
    assert after_wide <= 1.25 * fresh, (fresh, after_wide)
