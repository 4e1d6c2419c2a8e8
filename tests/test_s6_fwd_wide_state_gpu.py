"""GPU parity of the S6 forward with more than 16 states (17 to 64: the state
dimension N of the selective SSM is a free size of the model, "Mamba: Linear-
Time Sequence Modeling with Selective State Spaces", sec. 3.2).  Each row keeps
its states in 32 or 64 slots (four lanes of eight or sixteen); the slots past N
must add nothing.  Checked against the oracle for every form (exponential Euler,
zero-order hold, trapezoid), with an initial and a final state, on ragged
shapes (a partial row block, a short last tile, N that fills no slot group),
through the segmented plan (few rows, long sequence), the chained plan (enough
rows to fill the GPU, bit for bit against the pass without a workspace), the
allocation-free entry point and the host-buffer entry point.

Tolerances (max |gpu - ref| / (1 + |ref|)): 1e-4 with fp32 inputs, 2e-3 with
bf16 inputs (the oracle consumes the same bf16-rounded values)."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs, s6_inputs_torch
from helpers import max_rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-3


def _dev(inp, bf16):
    return {k: (to_dev(inp[k], bf16) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C")}


def _run(inp, bf16, h0=None, disc=0):
    import selective_state_space_160_b300 as msc
    d = _dev(inp, bf16)
    y, hl = msc.msc_selective_scan_fwd(d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                       d["z"], to_dev(inp["delta_bias"]),
                                       h0=None if h0 is None else to_dev(h0), return_last_state=True, disc=disc)
    return y.cpu().numpy(), hl.cpu().numpy()


def _ref(inp, h0=None, disc=0):
    return oracle.s6_fwd_disc(disc, inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                              inp["delta_bias"], h0=h0, return_last_state=True)


@pytest.mark.parametrize("N", [17, 24, 32, 33, 48, 63, 64])
@pytest.mark.parametrize("bf16", [False, True])
def test_shapes_with_initial_and_final_state(N, bf16):
    """dim 37: a partial second row block; L 96 (bf16: three 32-step tiles) or
    100 (fp32: six full 16-step tiles and a 4-step tail)."""
    L = 96 if bf16 else 100
    inp = s6_inputs(2, 37, L, N, seed=17_000 + N + 100 * bf16, bf16=bf16)
    h0 = np.random.default_rng(N).standard_normal((2, 37, N)).astype(np.float32)
    y, hl = _run(inp, bf16, h0=h0)
    ry, rh = _ref(inp, h0=h0)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y, ry) <= tol
    assert max_rel_err(hl, rh) <= tol


@pytest.mark.parametrize("disc", [oracle.DISC_ZOH, oracle.DISC_TRAPEZOID])
@pytest.mark.parametrize("N,bf16", [(40, True), (64, False), (20, False)])
def test_discretisations(disc, N, bf16):
    inp = s6_inputs(2, 33, 160, N, seed=17_100 + 3 * N + disc, bf16=bf16)
    h0 = np.random.default_rng(disc).standard_normal((2, 33, N)).astype(np.float32)
    y, hl = _run(inp, bf16, h0=h0, disc=disc)
    ry, rh = _ref(inp, h0=h0, disc=disc)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y, ry) <= tol
    assert max_rel_err(hl, rh) <= tol


def test_optional_inputs_left_out():
    inp = s6_inputs(1, 40, 64, 50, seed=17_200, with_z=False, with_D=False, with_bias=False)
    y, hl = _run(inp, False)
    ry, rh = _ref(inp)
    assert max_rel_err(y, ry) <= TOL_F32
    assert max_rel_err(hl, rh) <= TOL_F32


@pytest.mark.parametrize("N,L,bf16", [(64, 5000, False), (32, 6144, True)])
def test_long_sequence_segments(N, L, bf16):
    """Few rows: aggregate pass, carry pass and full pass over segments."""
    import selective_state_space_160_b300 as msc
    assert msc.msc_selective_scan_fwd_workspace_size(1, 3, L, N) > 0
    inp = s6_inputs(1, 3, L, N, seed=17_300 + N, bf16=bf16)
    h0 = np.random.default_rng(3).standard_normal((1, 3, N)).astype(np.float32)
    y, hl = _run(inp, bf16, h0=h0)
    ry, rh = _ref(inp, h0=h0)
    tol = TOL_BF16 if bf16 else TOL_F32
    assert max_rel_err(y, ry) <= tol
    assert max_rel_err(hl, rh) <= tol


@pytest.mark.parametrize("N,dim,L", [(64, 9500, 1024), (32, 9473, 2000)])
def test_chained_equals_single_pass_bitwise(N, dim, L):
    """Enough row blocks (297 or more) for the chained plan with 32 or 64 state
    slots: persistent CTAs hand the state of each row block from chunk to chunk;
    the result equals the pass without a workspace bit for bit, and sampled rows
    (the partial last block among them) match the oracle."""
    import torch
    import selective_state_space_160_b300 as msc
    batch = 1
    lib = msc.load_library()
    need = msc.msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    slots = 32 if N <= 32 else 64
    assert need >= batch * dim * slots * 4  # the chained plan's state hand-over
    inp = s6_inputs_torch(batch, dim, L, N, seed=17_400 + N, bf16=True)
    g = torch.Generator(device="cuda").manual_seed(11)
    h0 = torch.randn((batch, dim, N), device="cuda", generator=g)
    buf = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    ws = buf[off:off + need]
    ptr = lambda t: None if t is None else t.data_ptr()
    outs = []
    for w in (ws, None):
        y = torch.full((batch, dim, L), float("nan"), dtype=torch.float32, device="cuda")
        hl = torch.full((batch, dim, N), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.msc_selective_scan_fwd(batch, dim, L, N, 1, ptr(inp["u"]), ptr(inp["delta"]), ptr(inp["A"]),
                                        ptr(inp["B"]), ptr(inp["C"]), ptr(inp["D"]), ptr(inp["z"]),
                                        ptr(inp["delta_bias"]), ptr(h0), ptr(y), ptr(hl),
                                        None if w is None else w.data_ptr(), 0 if w is None else need,
                                        torch.cuda.current_stream().cuda_stream)
        assert st == 0, msc.msc_last_error()
        outs.append((y, hl))
    torch.cuda.synchronize()
    msc.msc_check_device_status()
    (yc, hc), (ys, hs) = outs
    assert bool(torch.isfinite(yc).all())
    assert bool(torch.equal(yc, ys)) and bool(torch.equal(hc, hs))
    host = {k: inp[k].float().cpu().numpy() for k in ("B", "C")}
    for d in (0, 33, dim // 2, dim - 1):
        sub = {k: inp[k][:, d:d + 1, :].float().cpu().numpy() for k in ("u", "delta", "z")}
        ry, rh = oracle.s6_fwd(sub["u"], sub["delta"], inp["A"][d:d + 1].cpu().numpy(), host["B"], host["C"],
                               inp["D"][d:d + 1].cpu().numpy(), sub["z"], inp["delta_bias"][d:d + 1].cpu().numpy(),
                               h0=h0[:, d:d + 1].cpu().numpy(), return_last_state=True)
        assert max_rel_err(yc[:, d:d + 1].cpu().numpy(), ry) <= TOL_BF16, d
        assert max_rel_err(hc[:, d:d + 1].cpu().numpy(), rh) <= TOL_BF16, d
    del inp, yc, ys, buf
    torch.cuda.empty_cache()


def test_noalloc_entry_point():
    import torch
    import selective_state_space_160_b300 as msc
    batch, dim, L, N = 1, 8, 8192, 48
    inp = s6_inputs(batch, dim, L, N, seed=17_500)
    d = _dev(inp, False)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y = torch.empty((batch, dim, L), dtype=torch.float32, device="cuda")
    hl = torch.empty((batch, dim, N), dtype=torch.float32, device="cuda")
    lib = msc.load_library()
    st = lib.msc_selective_scan_fwd_noalloc(batch, dim, L, N, 0, d["u"].data_ptr(), d["delta"].data_ptr(),
                                            A.data_ptr(), d["B"].data_ptr(), d["C"].data_ptr(), D.data_ptr(),
                                            d["z"].data_ptr(), bias.data_ptr(), None, y.data_ptr(),
                                            hl.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, msc.msc_last_error()
    ry, rh = _ref(inp)
    assert max_rel_err(y.cpu().numpy(), ry) <= TOL_F32
    assert max_rel_err(hl.cpu().numpy(), rh) <= TOL_F32


def test_host_buffer_entry_point():
    import torch
    import selective_state_space_160_b300 as msc
    inp = s6_inputs(3, 40, 256, 32, seed=17_600, bf16=True)
    h = {}
    for k in ("u", "delta", "z", "B", "C"):
        h[k] = torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(torch.bfloat16).pin_memory()
    y = msc.msc_selective_scan_fwd_host(h["u"], h["delta"], to_dev(inp["A"]), h["B"], h["C"], to_dev(inp["D"]),
                                        h["z"], to_dev(inp["delta_bias"]), chunk_batch=1)
    torch.cuda.synchronize()
    yd, _ = _run(inp, True)
    assert np.array_equal(y.numpy(), yd)
    assert max_rel_err(y.numpy(), _ref(inp)[0]) <= TOL_BF16


@pytest.mark.parametrize("batch,dim,L,N,bf16,disc", [
    (2, 37, 61, 20, True, 0),       # bf16 rows of 122 bytes: padded to 64 steps
    (1, 33, 63, 64, False, 0),      # fp32 rows of 252 bytes
    (2, 5, 1003, 48, True, 0),      # few rows: segments over the padded length
    (1, 9500, 1001, 32, True, 0),   # enough rows for the chained plan
    (2, 20, 77, 40, False, 1),      # zero-order hold
    (1, 3, 1, 17, True, 0),         # a single step
])
def test_unaligned_rows_through_padded_copies(batch, dim, L, N, bf16, disc):
    """Rows whose byte stride is not a multiple of 16 are copied to a padded pitch
    in the workspace; delta's padded steps are -inf, so Delta is 0 there and the
    state passes them unchanged: y and h_last match the oracle."""
    import selective_state_space_160_b300 as msc
    assert msc.msc_selective_scan_fwd_workspace_size(batch, dim, L, N) > 0  # the padded copies are required
    inp = s6_inputs(batch, dim, L, N, seed=17_800 + L + N, bf16=bf16)
    h0 = np.random.default_rng(L).standard_normal((batch, dim, N)).astype(np.float32)
    d = _dev(inp, bf16)
    y, hl = msc.msc_selective_scan_fwd(d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                       d["z"], to_dev(inp["delta_bias"]), h0=to_dev(h0), return_last_state=True,
                                       disc=disc)
    msc.msc_check_device_status()
    tol = TOL_BF16 if bf16 else TOL_F32
    if dim > 100:  # sampled rows
        ds = [0, 33, dim // 2, dim - 1]
        sub = dict(inp)
        for k in ("u", "delta", "z"):
            sub[k] = inp[k][:, ds, :]
        sub["A"], sub["D"], sub["delta_bias"] = inp["A"][ds], inp["D"][ds], inp["delta_bias"][ds]
        ry, rh = oracle.s6_fwd_disc(disc, sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                                    sub["delta_bias"], h0=h0[:, ds], return_last_state=True)
        assert max_rel_err(y.cpu().numpy()[:, ds], ry) <= tol
        assert max_rel_err(hl.cpu().numpy()[:, ds], rh) <= tol
    else:
        ry, rh = _ref(inp, h0=h0, disc=disc)
        assert max_rel_err(y.cpu().numpy(), ry) <= tol
        assert max_rel_err(hl.cpu().numpy(), rh) <= tol


def test_wide_state_limits():
    """Above 16 states the trapezoid (whose carried half-term would enter a
    padded step) takes no unaligned rows, and the fused conv front end is not
    offered: both refused with MSC_ERR_UNSUPPORTED before any launch."""
    import torch
    import selective_state_space_160_b300 as msc
    inp = s6_inputs(1, 4, 63, 20, seed=17_700)
    d = _dev(inp, False)
    with pytest.raises(msc.MscError) as e:
        msc.msc_selective_scan_fwd(d["u"], d["delta"], to_dev(inp["A"]), d["B"], d["C"], to_dev(inp["D"]),
                                   d["z"], to_dev(inp["delta_bias"]), disc=msc.MSC_DISC_TRAPEZOID)
    assert "trapezoidal" in str(e.value)
    inp = s6_inputs(1, 4, 64, 20, seed=17_701)
    d = _dev(inp, False)
    w = torch.ones((4, 4), device="cuda")
    with pytest.raises(msc.MscError) as e:
        msc.msc_selective_scan_fwd_conv(d["u"], w, None, d["delta"], to_dev(inp["A"]), d["B"], d["C"],
                                        to_dev(inp["D"]), d["z"], to_dev(inp["delta_bias"]))
    assert "16" in str(e.value)
    msc.msc_check_device_status()
    torch.cuda.synchronize()


def test_noalloc_unaligned_rows():
    """The allocation-free entry point pads small problems inside its array."""
    import torch
    import selective_state_space_160_b300 as msc
    batch, dim, L, N = 1, 6, 45, 24
    inp = s6_inputs(batch, dim, L, N, seed=17_900)
    d = _dev(inp, False)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y = torch.empty((batch, dim, L), dtype=torch.float32, device="cuda")
    hl = torch.empty((batch, dim, N), dtype=torch.float32, device="cuda")
    st = msc.load_library().msc_selective_scan_fwd_noalloc(
        batch, dim, L, N, 0, d["u"].data_ptr(), d["delta"].data_ptr(), A.data_ptr(), d["B"].data_ptr(),
        d["C"].data_ptr(), D.data_ptr(), d["z"].data_ptr(), bias.data_ptr(), None, y.data_ptr(), hl.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, msc.msc_last_error()
    ry, rh = _ref(inp)
    assert max_rel_err(y.cpu().numpy(), ry) <= TOL_F32
    assert max_rel_err(hl.cpu().numpy(), rh) <= TOL_F32
