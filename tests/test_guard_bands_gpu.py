"""Guard bands around every output of every entry point: each output (and each
workspace, staging buffer and in-place state) is carved out of a larger device
allocation whose bytes before and after it hold a fixed pattern, and outputs
start as NaN.  After the call (through the C ABI, on ragged shapes: partial row
blocks, short last tiles and chunks, unaligned rows) the pattern must be intact
-- nothing was written outside the buffer -- and no NaN may remain in an
output -- every element was written.  This is the canary check of the failure
detection plan, run on the host after each call; it needs no device fault."""
import numpy as np
import pytest

from selective_state_space_160_b300.inputs import s6_inputs, ssd_inputs
from helpers import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device (or pinned host) tensor of `shape` inside a byte buffer with
    GUARD pattern bytes on each side, starting on an `align`-byte boundary."""

    def __init__(self, shape, dtype="float32", fill=float("nan"), host=False, align=256):
        import torch
        dt = getattr(torch, dtype)
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * torch.empty((), dtype=dt).element_size()
        raw = torch.full((2 * GUARD + self.nbytes + align,), PATTERN, dtype=torch.uint8,
                         device="cpu" if host else "cuda")
        if host:
            raw = raw.pin_memory()
        self.raw = raw
        self.off = GUARD + ((-(raw.data_ptr() + GUARD)) % align)
        self.t = raw[self.off:self.off + self.nbytes].view(dt).view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    @property
    def ptr(self):
        return self.t.data_ptr()

    def intact(self):
        import torch
        if self.raw.is_cuda:
            torch.cuda.synchronize()
        front = self.raw[:self.off]
        back = self.raw[self.off + self.nbytes:]
        return bool((front == PATTERN).all()) and bool((back == PATTERN).all())

    def written(self):
        import torch
        return not bool(torch.isnan(self.t.float()).any())


def _lib():
    import selective_state_space_160_b300 as msc
    return msc, msc.load_library()


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(outs, msc, st):
    assert st == 0, msc.msc_last_error()
    msc.msc_check_device_status()
    for name, g in outs.items():
        assert g.intact(), "write outside " + name
        if name not in ("workspace", "staging"):
            assert g.written(), name + " not fully written"


def _ptr(t):
    return None if t is None else t.data_ptr()


def _s6_dev(inp, bf16):
    return {k: (to_dev(inp[k], bf16) if inp[k] is not None else None) for k in ("u", "delta", "z", "B", "C")}


@pytest.mark.parametrize("batch,dim,L,N,bf16", [
    (2, 37, 96, 16, True),        # TMA path, partial row block
    (2, 37, 100, 16, False),      # fp32 16-step tiles, short last tile
    (1, 5, 63, 16, False),        # unaligned rows: plain-load kernel
    (2, 7, 61, 5, True),          # unaligned bf16 rows, N < 16
    (1, 3, 5000, 16, False),      # few rows, long: segmented plan (workspace required)
    (1, 3, 5000, 48, True),       # the same with 64 state slots
    (2, 37, 96, 33, False),       # 64 slots, partial row block
    (1, 24000, 1024, 16, True),   # chained plan (workspace optional, given)
])
def test_s6_forward(batch, dim, L, N, bf16):
    msc, lib = _lib()
    inp = s6_inputs(batch, dim, L, N, seed=31_000 + dim + L + N, bf16=bf16)
    d = _s6_dev(inp, bf16)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    h0 = to_dev(np.random.default_rng(N).standard_normal((batch, dim, N)).astype(np.float32))
    y = Guarded((batch, dim, L))
    hl = Guarded((batch, dim, N))
    outs = {"y": y, "h_last": hl}
    need = msc.msc_selective_scan_fwd_workspace_size(batch, dim, L, N)
    ws = None
    if need:
        ws = Guarded((need,), "uint8", fill=None)
        outs["workspace"] = ws
    st = lib.msc_selective_scan_fwd(batch, dim, L, N, 1 if bf16 else 0, _ptr(d["u"]), _ptr(d["delta"]), _ptr(A),
                                    _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), _ptr(h0),
                                    y.ptr, hl.ptr, ws.ptr if ws else None, need, _stream())
    _check(outs, msc, st)


@pytest.mark.parametrize("disc", [1, 2])
def test_s6_forward_discretisations(disc):
    msc, lib = _lib()
    batch, dim, L, N = 2, 33, 160, 20
    inp = s6_inputs(batch, dim, L, N, seed=31_100 + disc, bf16=True)
    d = _s6_dev(inp, True)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y, hl = Guarded((batch, dim, L)), Guarded((batch, dim, N))
    st = lib.msc_selective_scan_fwd_ex(batch, dim, L, N, 1, disc, _ptr(d["u"]), _ptr(d["delta"]), _ptr(A),
                                       _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), None,
                                       y.ptr, hl.ptr, None, 0, _stream())
    _check({"y": y, "h_last": hl}, msc, st)


@pytest.mark.parametrize("L", [96, 101])  # TMA kernel; plain-load kernel (unaligned rows)
def test_s6_forward_fused_conv(L):
    import torch
    msc, lib = _lib()
    batch, dim, N, K = 2, 37, 16, 4
    inp = s6_inputs(batch, dim, L, N, seed=31_200, bf16=True)
    d = _s6_dev(inp, True)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    g = torch.Generator(device="cuda").manual_seed(12)
    w = torch.randn((dim, K), device="cuda", generator=g) / 2.0
    cb = 0.1 * torch.randn(dim, device="cuda", generator=g)
    y, hl = Guarded((batch, dim, L)), Guarded((batch, dim, N))
    st = lib.msc_selective_scan_fwd_conv(batch, dim, L, N, K, 1, _ptr(d["u"]), w.data_ptr(), cb.data_ptr(),
                                         _ptr(d["delta"]), _ptr(A), _ptr(d["B"]), _ptr(d["C"]), _ptr(D),
                                         _ptr(d["z"]), _ptr(bias), None, y.ptr, hl.ptr, None, 0, _stream())
    _check({"y": y, "h_last": hl}, msc, st)


def test_s6_forward_noalloc():
    msc, lib = _lib()
    batch, dim, L, N = 1, 5, 9000, 16
    inp = s6_inputs(batch, dim, L, N, seed=31_300, bf16=True)
    d = _s6_dev(inp, True)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y, hl = Guarded((batch, dim, L)), Guarded((batch, dim, N))
    st = lib.msc_selective_scan_fwd_noalloc(batch, dim, L, N, 1, _ptr(d["u"]), _ptr(d["delta"]), _ptr(A),
                                            _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), None,
                                            y.ptr, hl.ptr, _stream())
    _check({"y": y, "h_last": hl}, msc, st)


def test_s6_forward_from_host_buffers():
    import torch
    msc, lib = _lib()
    batch, dim, L, N = 3, 37, 96, 16
    inp = s6_inputs(batch, dim, L, N, seed=31_400, bf16=True)
    h = {k: torch.from_numpy(np.ascontiguousarray(inp[k], dtype=np.float32)).to(torch.bfloat16).pin_memory()
         for k in ("u", "delta", "z", "B", "C")}
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y = Guarded((batch, dim, L), host=True)
    nst = lib.msc_selective_scan_fwd_host_staging_size(batch, dim, L, N, 1, 1, 2)
    stg = Guarded((nst,), "uint8", fill=None)
    st = lib.msc_selective_scan_fwd_host(batch, dim, L, N, 1, h["u"].data_ptr(), h["delta"].data_ptr(), _ptr(A),
                                         h["B"].data_ptr(), h["C"].data_ptr(), _ptr(D), h["z"].data_ptr(),
                                         _ptr(bias), y.ptr, 2, stg.ptr, nst, _stream())
    torch.cuda.synchronize()
    _check({"y": y, "staging": stg}, msc, st)


@pytest.mark.parametrize("batch,dim,L,bf16,N", [(2, 37, 64, True, 16), (1, 36, 48, False, 16),
                                                (2, 33, 2048, True, 16),
                                                (2, 37, 64, True, 40), (1, 9, 100, False, 64)])  # state slices
def test_s6_backward(batch, dim, L, bf16, N):
    import torch
    msc, lib = _lib()
    inp = s6_inputs(batch, dim, L, N, seed=31_500 + dim + L, bf16=bf16)
    d = _s6_dev(inp, bf16)
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    g = torch.Generator(device="cuda").manual_seed(13)
    dy = torch.randn((batch, dim, L), device="cuda", generator=g)
    dy = dy.to(torch.bfloat16) if bf16 else dy
    outs = {"du": Guarded((batch, dim, L)), "ddelta": Guarded((batch, dim, L)), "dA": Guarded((dim, N)),
            "dB": Guarded((batch, N, L)), "dC": Guarded((batch, N, L)), "dD": Guarded((dim,)),
            "dz": Guarded((batch, dim, L)), "ddelta_bias": Guarded((dim,))}
    need = msc.msc_selective_scan_bwd_workspace_size(batch, dim, L, N)
    ws = Guarded((need,), "uint8", fill=None)
    o = outs
    st = lib.msc_selective_scan_bwd(batch, dim, L, N, 1 if bf16 else 0, _ptr(d["u"]), _ptr(d["delta"]), _ptr(A),
                                    _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), dy.data_ptr(),
                                    o["du"].ptr, o["ddelta"].ptr, o["dA"].ptr, o["dB"].ptr, o["dC"].ptr,
                                    o["dD"].ptr, o["dz"].ptr, o["ddelta_bias"].ptr, ws.ptr, need, _stream())
    outs["workspace"] = ws
    _check(outs, msc, st)


@pytest.mark.parametrize("N,bf16", [(16, True), (5, False), (64, True), (40, False)])
def test_s6_decode_step(N, bf16):
    import torch
    msc, lib = _lib()
    batch, dim = 3, 37
    inp = s6_inputs(batch, dim, 1, N, seed=31_600 + N, bf16=bf16)
    d = {k: to_dev(inp[k][:, :, 0], bf16) for k in ("u", "delta", "z", "B", "C")}  # one step
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    state = Guarded((batch, dim, N), fill=0.5)
    y = Guarded((batch, dim))
    st = lib.msc_selective_state_update(batch, dim, N, 1 if bf16 else 0, _ptr(d["u"]), _ptr(d["delta"]), _ptr(A),
                                        _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), state.ptr,
                                        y.ptr, _stream())
    _check({"state": state, "y": y}, msc, st)
    torch.cuda.synchronize()


@pytest.mark.parametrize("L,width,bf16", [(96, 4, True), (61, 3, False), (130, 8, True)])
def test_causal_conv1d(L, width, bf16):
    import torch
    msc, lib = _lib()
    batch, dim = 2, 37
    g = torch.Generator(device="cuda").manual_seed(14 + width)
    x = torch.randn((batch, dim, L), device="cuda", generator=g)
    x = x.to(torch.bfloat16) if bf16 else x
    w = torch.randn((dim, width), device="cuda", generator=g) / 2.0
    cb = 0.1 * torch.randn(dim, device="cuda", generator=g)
    dt = 1 if bf16 else 0
    out = Guarded((batch, dim, L))
    st = lib.msc_causal_conv1d_fwd(batch, dim, L, width, dt, 0, x.data_ptr(), w.data_ptr(), cb.data_ptr(), 1,
                                   out.ptr, _stream())
    _check({"out": out}, msc, st)
    outb = Guarded((batch, dim, L), "bfloat16")
    st = lib.msc_causal_conv1d_fwd(batch, dim, L, width, dt, 1, x.data_ptr(), w.data_ptr(), cb.data_ptr(), 1,
                                   outb.ptr, _stream())
    _check({"out_bf16": outb}, msc, st)
    dout = torch.randn((batch, dim, L), device="cuda", generator=g)
    o = {"dx": Guarded((batch, dim, L)), "dweight": Guarded((dim, width)), "dbias": Guarded((dim,))}
    st = lib.msc_causal_conv1d_bwd(batch, dim, L, width, dt, x.data_ptr(), w.data_ptr(), cb.data_ptr(), 1,
                                   dout.data_ptr(), o["dx"].ptr, o["dweight"].ptr, o["dbias"].ptr, _stream())
    _check(o, msc, st)
    cs = Guarded((batch, dim, width - 1), fill=0.25) if width > 1 else None
    xt = x[:, :, 0].contiguous()
    y1 = Guarded((batch, dim))
    st = lib.msc_causal_conv1d_update(batch, dim, width, dt, 0, xt.data_ptr(), w.data_ptr(), cb.data_ptr(), 1,
                                      cs.ptr if cs else None, y1.ptr, _stream())
    _check({"y": y1, **({"conv_state": cs} if cs else {})}, msc, st)


@pytest.mark.parametrize("L,H,G,chunk,with_z", [(300, 20, 1, 256, True), (130, 3, 1, 64, False),
                                                 (512, 32, 2, 128, True)])
def test_ssd_forward_and_backward(L, H, G, chunk, with_z):
    msc, lib = _lib()
    batch, P, N = 1, 64, 128
    inp = ssd_inputs(batch, L, H, P, N, G, seed=31_700 + L + H, bf16=True, with_z=with_z, with_dy=True)
    d = {k: (to_dev(inp[k], True) if inp.get(k) is not None else None) for k in ("x", "delta", "B", "C", "z", "dy")}
    A, D, bias = to_dev(inp["A"]), to_dev(inp["D"]), to_dev(inp["delta_bias"])
    y, fs = Guarded((batch, L, H, P)), Guarded((batch, H, P, N))
    need = msc.msc_ssd_chunked_fwd_workspace_size(batch, L, H, P, N, G, chunk)
    ws = Guarded((need,), "uint8", fill=None, align=1024)  # the SSD workspace is 1024-byte aligned
    st = lib.msc_ssd_chunked_fwd(batch, L, H, P, N, G, chunk, 1, _ptr(d["x"]), _ptr(d["delta"]), _ptr(A),
                                 _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), y.ptr, fs.ptr,
                                 ws.ptr, need, _stream())
    _check({"y": y, "final_state": fs, "workspace": ws}, msc, st)
    o = {"dx": Guarded((batch, L, H, P)), "ddelta": Guarded((batch, L, H)), "dA": Guarded((H,)),
         "dB": Guarded((batch, L, G, N)), "dC": Guarded((batch, L, G, N)), "dD": Guarded((H,)),
         "ddelta_bias": Guarded((H,))}
    if with_z:
        o["dz"] = Guarded((batch, L, H, P))
    need = msc.msc_ssd_chunked_bwd_workspace_size(batch, L, H, P, N, G, chunk, int(with_z))
    wsb = Guarded((need,), "uint8", fill=None, align=1024)
    st = lib.msc_ssd_chunked_bwd(batch, L, H, P, N, G, chunk, 1, _ptr(d["x"]), _ptr(d["delta"]), _ptr(A),
                                 _ptr(d["B"]), _ptr(d["C"]), _ptr(D), _ptr(d["z"]), _ptr(bias), _ptr(d["dy"]),
                                 o["dx"].ptr, o["ddelta"].ptr, o["dA"].ptr, o["dB"].ptr, o["dC"].ptr, o["dD"].ptr,
                                 o["dz"].ptr if with_z else None, o["ddelta_bias"].ptr, wsb.ptr, need, _stream())
    o["workspace"] = wsb
    _check(o, msc, st)
