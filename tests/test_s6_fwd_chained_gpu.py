"""GPU tests of the S6 forward's chained schedule: with enough rows to fill the
GPU and sequences of 512 steps or more, persistent CTAs run each 32-row block
in time chunks and hand the state from chunk to chunk through the workspace.
The hand-over is an exact fp32 copy, so the chained pass must equal the pass
without a workspace (one CTA per row block) bit for bit, for every form that
runs through it (exponential Euler, zero-order hold, trapezoid, the fused conv
front end), with an initial state and the final state, on ragged shapes (a
partial last row block, a last chunk shorter than the others, fp32 inputs with
16-step tiles).  Sampled rows are also checked against the oracle."""
import numpy as np
import pytest

from oracle import oracle
from selective_state_space_160_b300.inputs import s6_inputs_torch
from helpers import max_rel_err

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-3

# (batch, dim, L, bf16): rows = batch * dim >= 23 680 make 740+ row blocks, the
# chained schedule's threshold on 148 SMs; dim % 32 != 0 leaves a partial last
# block; L = 2000 gives chunks of 512, 512, 512 and 464 steps
SHAPES = [(1, 24000, 1024, True), (2, 12013, 2000, True), (1, 24576, 1028, False)]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call(inp, batch, dim, L, N, bf16, y, h0=None, h_last=None, workspace=None, disc=0, conv=None):
    """The C entry point directly, so that the workspace can be left out."""
    import torch
    import selective_state_space_160_b300 as msc
    lib = msc.load_library()
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (workspace.data_ptr(), workspace.numel())
    stream = torch.cuda.current_stream().cuda_stream
    dt = 1 if bf16 else 0
    if conv is not None:
        w, cb = conv
        st = lib.msc_selective_scan_fwd_conv(batch, dim, L, N, w.shape[1], dt, _ptr(inp["u"]), _ptr(w), _ptr(cb),
                                             _ptr(inp["delta"]), _ptr(inp["A"]), _ptr(inp["B"]), _ptr(inp["C"]),
                                             _ptr(inp["D"]), _ptr(inp["z"]), _ptr(inp["delta_bias"]), _ptr(h0),
                                             _ptr(y), _ptr(h_last), ws_ptr, ws_bytes, stream)
    else:
        st = lib.msc_selective_scan_fwd_ex(batch, dim, L, N, dt, disc, _ptr(inp["u"]), _ptr(inp["delta"]),
                                           _ptr(inp["A"]), _ptr(inp["B"]), _ptr(inp["C"]), _ptr(inp["D"]),
                                           _ptr(inp["z"]), _ptr(inp["delta_bias"]), _ptr(h0), _ptr(y),
                                           _ptr(h_last), ws_ptr, ws_bytes, stream)
    assert st == 0, msc.msc_last_error()


def _workspace(batch, dim, L, N):
    import torch
    import selective_state_space_160_b300 as msc
    need = msc.msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    assert need > 0  # the chained schedule's scratch
    buf = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    return buf[off:off + need]


def _pair(inp, batch, dim, L, N, bf16, **kw):
    """y and h_last of the chained pass and of the pass without a workspace."""
    import torch
    out = []
    for ws in (_workspace(batch, dim, L, N), None):
        y = torch.full((batch, dim, L), float("nan"), dtype=torch.float32, device="cuda")
        hl = torch.full((batch, dim, N), float("nan"), dtype=torch.float32, device="cuda")
        _call(inp, batch, dim, L, N, bf16, y, h_last=hl, workspace=ws, **kw)
        out.append((y, hl))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("batch,dim,L,bf16", SHAPES)
def test_chained_equals_single_pass_bitwise_and_oracle(batch, dim, L, bf16):
    import torch
    import selective_state_space_160_b300 as msc
    N = 16
    inp = s6_inputs_torch(batch, dim, L, N, seed=5100 + dim + L, bf16=bf16)
    g = torch.Generator(device="cuda").manual_seed(9)
    h0 = torch.randn((batch, dim, N), device="cuda", generator=g)
    (yc, hc), (ys, hs) = _pair(inp, batch, dim, L, N, bf16, h0=h0)
    msc.msc_check_device_status()
    assert bool(torch.equal(yc, ys)) and bool(torch.equal(hc, hs))
    assert bool(torch.isfinite(yc).all())
    # sampled rows, the partial last block included, against the oracle
    host = {k: inp[k].float().cpu().numpy() for k in ("B", "C")}
    for b in range(batch):
        for d in (0, 31, 32, dim // 2, dim - 1):
            sub = {k: inp[k][b:b + 1, d:d + 1, :].float().cpu().numpy() for k in ("u", "delta", "z")}
            ry, rh = oracle.s6_fwd(sub["u"], sub["delta"], inp["A"][d:d + 1].cpu().numpy(), host["B"][b:b + 1],
                                   host["C"][b:b + 1], inp["D"][d:d + 1].cpu().numpy(), sub["z"],
                                   inp["delta_bias"][d:d + 1].cpu().numpy(),
                                   h0=h0[b:b + 1, d:d + 1].cpu().numpy(), return_last_state=True)
            tol = TOL_BF16 if bf16 else TOL_F32
            assert max_rel_err(yc[b:b + 1, d:d + 1].cpu().numpy(), ry) <= tol, (b, d)
            assert max_rel_err(hc[b:b + 1, d:d + 1].cpu().numpy(), rh) <= tol, (b, d)
    del inp, yc, ys
    torch.cuda.empty_cache()


@pytest.mark.parametrize("disc", [1, 2])
def test_chained_discretisations_bitwise(disc):
    """Zero-order hold (1) and trapezoid (2): the trapezoid carries the previous
    step's input term, which a chunk rebuilds from the step before it."""
    import torch
    batch, dim, L, N = 2, 12013, 2000, 16
    inp = s6_inputs_torch(batch, dim, L, N, seed=5200 + disc, bf16=True)
    (yc, hc), (ys, hs) = _pair(inp, batch, dim, L, N, True, disc=disc)
    assert bool(torch.equal(yc, ys)) and bool(torch.equal(hc, hs))
    # and against the oracle on a few rows
    host = {k: inp[k].float().cpu().numpy() for k in ("B", "C")}
    for d in (0, 6000, dim - 1):
        sub = {k: inp[k][:, d:d + 1, :].float().cpu().numpy() for k in ("u", "delta", "z")}
        ry = oracle.s6_fwd_disc(disc, sub["u"], sub["delta"], inp["A"][d:d + 1].cpu().numpy(), host["B"],
                                host["C"], inp["D"][d:d + 1].cpu().numpy(), sub["z"],
                                inp["delta_bias"][d:d + 1].cpu().numpy())
        assert max_rel_err(yc[:, d:d + 1].cpu().numpy(), ry) <= TOL_BF16, d
    del inp, yc, ys
    torch.cuda.empty_cache()


def test_chained_fused_conv_bitwise():
    """The fused causal conv1d front end reads the three inputs before a chunk
    from memory; chained and single-pass results agree bit for bit."""
    import torch
    batch, dim, L, N, K = 1, 24000, 1024, 16, 4
    inp = s6_inputs_torch(batch, dim, L, N, seed=5300, bf16=True)
    g = torch.Generator(device="cuda").manual_seed(10)
    w = torch.randn((dim, K), device="cuda", generator=g) / 2.0
    cb = 0.1 * torch.randn(dim, device="cuda", generator=g)
    (yc, hc), (ys, hs) = _pair(inp, batch, dim, L, N, True, conv=(w, cb))
    assert bool(torch.equal(yc, ys)) and bool(torch.equal(hc, hs))
    d = 7
    x = inp["u"][:, d:d + 1, :].float().cpu().numpy()
    u = oracle.causal_conv1d(x, w[d:d + 1].cpu().numpy(), cb[d:d + 1].cpu().numpy(), silu=True)
    ry = oracle.s6_fwd(u, inp["delta"][:, d:d + 1].float().cpu().numpy(), inp["A"][d:d + 1].cpu().numpy(),
                       inp["B"].float().cpu().numpy(), inp["C"].float().cpu().numpy(),
                       inp["D"][d:d + 1].cpu().numpy(), inp["z"][:, d:d + 1].float().cpu().numpy(),
                       inp["delta_bias"][d:d + 1].cpu().numpy())
    assert max_rel_err(yc[:, d:d + 1].cpu().numpy(), ry) <= TOL_BF16
    del inp, yc, ys
    torch.cuda.empty_cache()
