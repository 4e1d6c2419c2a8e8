"""Host-only checks of the C ABI: the library loads, exports every symbol that
include/msc.h declares, and rejects bad arguments before launching anything.
No test here needs a GPU (no compute call reaches a kernel)."""
import ctypes
import os
import re
import subprocess

import pytest

import selective_state_space_160_b300 as msc
from selective_state_space_160_b300 import build as msc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    msc_build.build()
    return msc.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "msc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msc_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("msc_selective_scan_fwd", "msc_selective_scan_bwd", "msc_ssd_chunked_fwd",
              "msc_check_device_status", "msc_status_string", "msc_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", msc.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (msc_[a-z0-9_]+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # the python binding declares a signature for every exported entry point
    assert set(declared_functions()) <= set(msc.SIGNATURES)


def test_status_strings(lib):
    assert msc.msc_status_string(0) == "MSC_OK"
    assert msc.msc_status_string(4) == "MSC_ERR_TIMEOUT"
    assert msc.msc_status_string(99) == "MSC_ERR_UNKNOWN"


def _fwd(lib, **kw):
    args = dict(batch=1, dim=4, L=64, N=16, dt=0, u=16, delta=16, A=16, B=16, C=16, D=None, z=None,
                bias=None, h0=None, y=16, hl=None, ws=None, wsb=0)
    args.update(kw)
    return lib.msc_selective_scan_fwd(args["batch"], args["dim"], args["L"], args["N"], args["dt"],
                                      args["u"], args["delta"], args["A"], args["B"], args["C"],
                                      args["D"], args["z"], args["bias"], args["h0"], args["y"],
                                      args["hl"], args["ws"], args["wsb"], None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, u=None) == msc.MSC_ERR_INVALID_ARG
    assert "u must not be NULL" in msc.msc_last_error()
    assert _fwd(lib, y=None) == msc.MSC_ERR_INVALID_ARG
    assert _fwd(lib, u=18) == msc.MSC_ERR_INVALID_ARG          # misaligned
    assert "aligned" in msc.msc_last_error()
    assert _fwd(lib, L=0) == msc.MSC_ERR_INVALID_ARG
    assert _fwd(lib, batch=-1) == msc.MSC_ERR_INVALID_ARG
    assert _fwd(lib, dt=7) == msc.MSC_ERR_INVALID_ARG
    assert _fwd(lib, N=65) == msc.MSC_ERR_UNSUPPORTED
    assert _fwd(lib, N=0) == msc.MSC_ERR_UNSUPPORTED
    # 17..64 states stream through TMA only: rows of 63 fp32 steps (252 bytes)
    # are copied to a padded pitch in the workspace, which is then required
    need = msc.msc_selective_scan_fwd_workspace_size(1, 4, 63, 17)
    assert need >= 4 * (4 * 64 * 4) + 2 * (17 * 64 * 4)  # u, delta, z, y and B, C at a pitch of 64
    assert _fwd(lib, N=17, L=63) == msc.MSC_ERR_WORKSPACE
    # the trapezoid cannot take padded steps: refused before any launch
    st = lib.msc_selective_scan_fwd_ex(1, 4, 63, 17, 0, 2, 16, 16, 16, 16, 16, None, None, None, None, 16, None,
                                       4096, need, None)
    assert st == msc.MSC_ERR_UNSUPPORTED and "trapezoidal" in msc.msc_last_error()
    assert _fwd(lib, z=20) == msc.MSC_ERR_INVALID_ARG


def test_fwd_workspace_query_and_check(lib):
    # plenty of rows: the chained schedule's state hand-over (optional: without it
    # one CTA per row block) -- 40960 rows x 16 states x 4 B, plus a 256-byte
    # control block and one 4-byte flag per 32-row block
    need = msc.msc_selective_scan_fwd_workspace_size(8, 5120, 2048, 16)
    assert 40960 * 16 * 4 + 256 + 1280 * 4 <= need <= 40960 * 16 * 4 + 256 + 1280 * 4 + 256
    # a short sequence with one row block: one item, no workspace
    assert msc.msc_selective_scan_fwd_workspace_size(1, 64, 256, 16) == 0
    # few rows and a long sequence: segments need a workspace
    need = msc.msc_selective_scan_fwd_workspace_size(1, 1536, 1 << 20, 16)
    assert need > 0
    assert _fwd(lib, batch=1, dim=1536, L=1 << 20) == msc.MSC_ERR_WORKSPACE
    assert _fwd(lib, batch=1, dim=1536, L=1 << 20, ws=4096, wsb=need - 1) == msc.MSC_ERR_WORKSPACE
    assert msc.msc_selective_scan_fwd_workspace_size(0, 4, 4, 4) == 0
    # 32 and 64 state slots: the hand-over holds every slot; 65 states: no plan
    for N, slots in ((17, 32), (32, 32), (33, 64), (64, 64)):
        need = msc.msc_selective_scan_fwd_workspace_size(8, 5120, 2048, N)
        assert 40960 * slots * 4 + 256 + 1280 * 4 <= need <= 40960 * slots * 4 + 256 + 1280 * 4 + 256, N
    assert msc.msc_selective_scan_fwd_workspace_size(8, 5120, 2048, 65) == 0
    assert msc.msc_selective_scan_fwd_workspace_size(1, 1536, 1 << 20, 64) > 0


def test_bwd_rejects_bad_arguments(lib):
    f = lib.msc_selective_scan_bwd
    ok = [16] * 5
    # dD must accompany D
    st = f(1, 4, 64, 16, 0, *ok, 16, None, None, 16, 16, 16, 16, 16, 16, None, None, None, None, 0, None)
    assert st == msc.MSC_ERR_INVALID_ARG and "dD" in msc.msc_last_error()
    st = f(1, 4, 64, 16, 0, *ok, None, 16, None, 16, 16, 16, 16, 16, 16, None, None, None, None, 0, None)
    assert st == msc.MSC_ERR_INVALID_ARG and "dz" in msc.msc_last_error()
    st = f(1, 4, 64, 16, 0, *ok, None, None, None, None, 16, 16, 16, 16, 16, None, None, None, None, 0, None)
    assert st == msc.MSC_ERR_INVALID_ARG and "dy" in msc.msc_last_error()
    # rows of 2^31 steps do not fit the 32-bit TMA coordinates: refused before any device work
    big = 1 << 31
    ws = msc.msc_selective_scan_bwd_workspace_size(1, 4, big, 16)
    st = f(1, 4, big, 16, 1, *ok, None, None, None, 16, 16, 16, 16, 16, 16, None, None, None, 4096, ws, None)
    assert st == msc.MSC_ERR_UNSUPPORTED and "2^31" in msc.msc_last_error()
    # up to 64 states, as the forward; above 16 the workspace also holds one
    # 16-state slice of A and of dA
    st = f(1, 4, 64, 65, 0, *ok, None, None, None, 16, 16, 16, 16, 16, 16, None, None, None, None, 0, None)
    assert st == msc.MSC_ERR_UNSUPPORTED and "[1, 64]" in msc.msc_last_error()
    assert msc.msc_selective_scan_bwd_workspace_size(1, 4, 64, 65) == 0
    w16 = msc.msc_selective_scan_bwd_workspace_size(1, 4, 64, 16)
    assert msc.msc_selective_scan_bwd_workspace_size(1, 4, 64, 17) == w16 + 2 * 256
    assert msc.msc_selective_scan_bwd_workspace_size(1, 4, 64, 64) == w16 + 2 * 256
    # a smaller workspace above 16 states is refused before any launch
    st = f(1, 4, 64, 40, 0, *ok, None, None, None, 16, 16, 16, 16, 16, 16, None, None, None, 4096, w16, None)
    assert st == msc.MSC_ERR_WORKSPACE


def test_ssd_rejects_bad_arguments(lib):
    f = lib.msc_ssd_chunked_fwd

    def call(b=1, L=256, H=4, P=64, N=128, G=1, Q=256, dt=1, ws=1024, wsb=1 << 30):
        return f(b, L, H, P, N, G, Q, dt, 16, 16, 16, 16, 16, None, None, None, 16, None, ws, wsb, None)

    assert call(G=3) == msc.MSC_ERR_INVALID_ARG
    assert call(P=32) == msc.MSC_ERR_UNSUPPORTED
    assert call(N=64) == msc.MSC_ERR_UNSUPPORTED
    assert call(Q=100) == msc.MSC_ERR_UNSUPPORTED
    assert call(dt=0) == msc.MSC_ERR_UNSUPPORTED
    assert call(ws=None, wsb=0) == msc.MSC_ERR_WORKSPACE
    assert call(ws=2048 + 16) == msc.MSC_ERR_INVALID_ARG        # workspace misaligned
    assert call(ws=2048 + 256) == msc.MSC_ERR_INVALID_ARG       # 256-byte aligned is not enough: 1024
    assert "1024-byte" in msc.msc_last_error()


def test_check_device_status_null_workspace_signature(lib):
    # only the signature is checked here; calling it needs a CUDA context
    assert lib.msc_check_device_status.restype == ctypes.c_int


def test_step_rejects_bad_arguments(lib):
    f = lib.msc_selective_state_update

    def call(batch=2, dim=4, N=16, dt=1, u=16, state=16, y=16, z=None):
        return f(batch, dim, N, dt, u, 16, 16, 16, 16, None, z, None, state, y, None)

    assert call(state=None) == msc.MSC_ERR_INVALID_ARG
    assert "state must not be NULL" in msc.msc_last_error()
    assert call(y=None) == msc.MSC_ERR_INVALID_ARG
    assert call(u=24) == msc.MSC_ERR_INVALID_ARG                 # misaligned
    assert call(z=40) == msc.MSC_ERR_INVALID_ARG
    assert call(N=65) == msc.MSC_ERR_UNSUPPORTED                 # up to 64 states
    assert call(N=0) == msc.MSC_ERR_UNSUPPORTED
    assert call(dim=0) == msc.MSC_ERR_INVALID_ARG
    assert call(dt=5) == msc.MSC_ERR_INVALID_ARG


def test_conv1d_rejects_bad_arguments(lib):
    f = lib.msc_causal_conv1d_fwd

    def call(batch=1, dim=4, L=16, K=4, idt=1, odt=1, x=16, w=16, out=16):
        return f(batch, dim, L, K, idt, odt, x, w, None, 1, out, None)

    assert call(x=None) == msc.MSC_ERR_INVALID_ARG
    assert call(K=9) == msc.MSC_ERR_UNSUPPORTED
    assert call(K=0) == msc.MSC_ERR_UNSUPPORTED
    assert call(odt=3) == msc.MSC_ERR_INVALID_ARG
    assert call(L=0) == msc.MSC_ERR_INVALID_ARG
    assert call(out=24) == msc.MSC_ERR_INVALID_ARG
    g = lib.msc_causal_conv1d_update
    assert g(1, 4, 4, 1, 1, 16, 16, None, 1, None, 16, None) == msc.MSC_ERR_INVALID_ARG   # state required
    assert "conv_state" in msc.msc_last_error()


def test_fwd_ex_rejects_bad_arguments(lib):
    f = lib.msc_selective_scan_fwd_ex

    def call(L=64, dt=1, disc=1, N=16, ws=None, wsb=0):
        return f(1, 4, L, N, dt, disc, 16, 16, 16, 16, 16, None, None, None, None, 16, None, ws, wsb, None)

    assert call(disc=7) == msc.MSC_ERR_INVALID_ARG
    assert "disc" in msc.msc_last_error()
    # rows that TMA cannot stream: up to 16 states the plain-load kernel takes
    # every form (a GPU test covers it); above, the padded copies need the
    # workspace, and the trapezoid cannot take padded steps at all
    assert call(L=63, N=20, disc=msc.MSC_DISC_ZOH) == msc.MSC_ERR_WORKSPACE
    need = msc.msc_selective_scan_fwd_workspace_size(1, 4, 66, 20)
    assert call(L=66, dt=1, N=20, disc=msc.MSC_DISC_TRAPEZOID, ws=4096, wsb=need) == msc.MSC_ERR_UNSUPPORTED
    # rows of 2^31 steps do not fit the 32-bit TMA coordinates, and above 16
    # states only the TMA kernel runs: refused before any launch
    big = 1 << 31
    ws = msc.msc_selective_scan_fwd_workspace_size(1, 4, big, 20)
    r = f(1, 4, big, 20, 1, msc.MSC_DISC_ZOH, 16, 16, 16, 16, 16, None, None, None, None, 16, None, 4096, ws, None)
    assert r == msc.MSC_ERR_UNSUPPORTED and "2^31" in msc.msc_last_error()


def test_ssd_bwd_rejects_bad_arguments(lib):
    f = lib.msc_ssd_chunked_bwd

    def call(b=1, L=256, H=4, P=64, N=128, G=1, Q=256, dt=1, D=None, z=None, bias=None, dy=16,
             dD=None, dz=None, dbias=None, ws=1024, wsb=1 << 30):
        return f(b, L, H, P, N, G, Q, dt, 16, 16, 16, 16, 16, D, z, bias, dy, 16, 16, 16, 16, 16,
                 dD, dz, dbias, ws, wsb, None)

    assert call(G=3) == msc.MSC_ERR_INVALID_ARG
    assert call(P=32) == msc.MSC_ERR_UNSUPPORTED
    assert call(Q=100) == msc.MSC_ERR_UNSUPPORTED
    assert call(dt=0) == msc.MSC_ERR_UNSUPPORTED
    assert call(H=24, G=2) == msc.MSC_ERR_UNSUPPORTED          # 12 heads per group
    assert call(dy=None) == msc.MSC_ERR_INVALID_ARG and "dy" in msc.msc_last_error()
    assert call(D=16) == msc.MSC_ERR_INVALID_ARG and "dD" in msc.msc_last_error()
    assert call(z=16) == msc.MSC_ERR_INVALID_ARG and "dz" in msc.msc_last_error()
    assert call(bias=16) == msc.MSC_ERR_INVALID_ARG and "ddelta_bias" in msc.msc_last_error()
    assert call(ws=None, wsb=0) == msc.MSC_ERR_WORKSPACE
    assert call(ws=2048 + 16) == msc.MSC_ERR_INVALID_ARG        # workspace misaligned
    assert call(ws=2048 + 256) == msc.MSC_ERR_INVALID_ARG       # 256-byte aligned is not enough: 1024
    assert "1024-byte" in msc.msc_last_error()
    # the gate needs room for the recomputed pre-gate output and the forward's workspace
    no_z = msc.msc_ssd_chunked_bwd_workspace_size(2, 1000, 8, 64, 128, 1, 256, False)
    with_z = msc.msc_ssd_chunked_bwd_workspace_size(2, 1000, 8, 64, 128, 1, 256, True)
    assert 0 < no_z < with_z
    assert call(z=16, dz=16, wsb=no_z, L=1000, b=2, H=8) == msc.MSC_ERR_WORKSPACE


def test_signatures_match_header_argument_counts():
    """Every binding signature has as many arguments as the header declares."""
    src = open(os.path.join(ROOT, "include", "msc.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for name in declared_functions():
        m = re.search(r"\b%s\s*\(([^)]*)\)" % name, src)
        params = m.group(1).strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(msc.SIGNATURES[name][1]) == n, name


def test_fwd_conv_rejects_bad_arguments(lib):
    f = lib.msc_selective_scan_fwd_conv

    def call(K=4, L=64, dt=1, x=16, w=16, N=16):
        return f(1, 4, L, N, K, dt, x, w, None, 16, 16, 16, 16, None, None, None, None, 16, None, None, 0, None)

    assert call(K=0) == msc.MSC_ERR_UNSUPPORTED
    assert call(K=5) == msc.MSC_ERR_UNSUPPORTED
    assert call(x=None) == msc.MSC_ERR_INVALID_ARG and "x" in msc.msc_last_error()
    assert call(w=None) == msc.MSC_ERR_INVALID_ARG and "conv_weight" in msc.msc_last_error()
    assert call(N=17) == msc.MSC_ERR_UNSUPPORTED                # up to 16 states
    assert call(L=100, N=17) == msc.MSC_ERR_UNSUPPORTED         # at any seqlen


def test_conv1d_bwd_rejects_bad_arguments(lib):
    f = lib.msc_causal_conv1d_bwd

    def call(batch=1, dim=4, L=16, K=4, idt=1, x=16, w=16, dout=16, dx=16, dw=16, db=None):
        return f(batch, dim, L, K, idt, x, w, None, 1, dout, dx, dw, db, None)

    assert call(dout=None) == msc.MSC_ERR_INVALID_ARG and "dout" in msc.msc_last_error()
    assert call(dx=None) == msc.MSC_ERR_INVALID_ARG and "dx" in msc.msc_last_error()
    assert call(dw=None) == msc.MSC_ERR_INVALID_ARG and "dweight" in msc.msc_last_error()
    assert call(x=None) == msc.MSC_ERR_INVALID_ARG
    assert call(dx=24) == msc.MSC_ERR_INVALID_ARG               # dx misaligned
    assert call(db=40) == msc.MSC_ERR_INVALID_ARG               # dbias misaligned
    assert call(K=9) == msc.MSC_ERR_UNSUPPORTED
    assert call(idt=3) == msc.MSC_ERR_INVALID_ARG
    assert call(batch=0) == msc.MSC_ERR_INVALID_ARG


def test_binding_has_no_cpu_path(monkeypatch):
    """The product path refuses host tensors (no CPU fallback) and raises when
    the library has not been built."""
    import torch
    x = torch.zeros((1, 4, 16))
    A = torch.zeros((4, 16))
    Bm = torch.zeros((1, 16, 16))
    with pytest.raises(ValueError, match="CUDA tensor"):
        msc.msc_selective_scan_fwd(x, x, A, Bm, Bm)
    with pytest.raises(ValueError, match="CUDA tensor"):
        msc.msc_causal_conv1d_fwd(x, torch.zeros((4, 4)))
    monkeypatch.setattr(msc, "_LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmsc.so"))
    monkeypatch.setattr(msc, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        msc.load_library()


def test_fwd_host_rejects_bad_arguments(lib):
    f = lib.msc_selective_scan_fwd_host

    def call(batch=2, L=64, dt=1, u=16, y=16, chunk=1, st=4096, stb=1 << 30):
        return f(batch, 4, L, 16, dt, u, 16, 16, 16, 16, None, None, None, y, chunk, st, stb, None)

    assert call(u=None) == msc.MSC_ERR_INVALID_ARG
    assert call(y=None) == msc.MSC_ERR_INVALID_ARG
    assert call(chunk=0) == msc.MSC_ERR_INVALID_ARG
    assert call(dt=5) == msc.MSC_ERR_INVALID_ARG
    assert call(st=None) == msc.MSC_ERR_WORKSPACE
    assert call(stb=16) == msc.MSC_ERR_WORKSPACE
    assert call(st=4096 + 16) == msc.MSC_ERR_INVALID_ARG           # staging misaligned
    one = lib.msc_selective_scan_fwd_host_staging_size(8, 4, 64, 16, 1, 1, 1)
    two = lib.msc_selective_scan_fwd_host_staging_size(8, 4, 64, 16, 1, 1, 2)
    assert 0 < one < two
    assert lib.msc_selective_scan_fwd_host_staging_size(8, 4, 64, 16, 1, 1, 0) == 0
