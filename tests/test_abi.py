"""The C-ABI library builds, loads and exports every function include/attn.h
declares; host-side argument checks return their codes (no GPU needed: every
call here fails validation before any CUDA call)."""
import ctypes

import pytest

from exact_io_aware_14_gb300 import build as native_build
from exact_io_aware_14_gb300 import _native


@pytest.fixture(scope="module")
def L():
    native_build.build()
    return _native.lib()


def test_header_declares_the_boundary():
    names = _native.declared_functions()
    for n in ("attn_fwd", "attn_fwd_splitkv", "attn_splitkv_workspace_size", "attn_get_device_status",
              "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _native.declared_functions():
        assert hasattr(L, name), name


def test_only_the_boundary_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH], capture_output=True, text=True).stdout
    ours = sorted({ln.split()[-1] for ln in out.splitlines() if " T attn_" in ln})
    assert ours == _native.declared_functions()


def test_status_strings(L):
    for code in range(8):
        s = _native.status_string(code)
        assert s and s != "unknown status"
    assert _native.status_string(99) == "unknown status"


def _fwd(L, **kw):
    a = dict(q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=2, Nq=8, Nk=8, d=64, causal=0, scale=0.125)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["o"]), vp(a["lse"]), a["B"], a["Hq"], a["Hkv"],
                      a["Nq"], a["Nk"], a["d"], a["causal"], a["scale"], None)


def test_attn_fwd_argument_checks(L):
    assert _fwd(L, Hq=3, Hkv=2) == 1          # heads do not divide
    assert _fwd(L, B=0) == 1
    assert _fwd(L, Nq=-1) == 1
    assert _fwd(L, causal=3) == 1             # 0 none, 1 top-left, 2 bottom-right
    assert _fwd(L, causal=-1) == 1
    assert _fwd(L, scale=float("nan")) == 1
    assert _fwd(L, scale=float("inf")) == 1
    assert _fwd(L, d=96) == 2                 # not built
    assert _fwd(L, q=0) == 1                  # NULL
    assert _fwd(L, q=8) == 3                  # misaligned
    assert _fwd(L, lse=2) == 3
    assert _fwd(L, Nq=0) == 0                 # empty: nothing to do


def _splitkv(L, **kw):
    a = dict(q=16, k=16, v=16, s=16, S=2048, o=16, lse=16, B=2, Hq=8, Hkv=2, d=128, scale=0.1, chunk=1024,
             ws=16, wsb=1 << 30)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd_splitkv(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["s"]), a["S"], vp(a["o"]), vp(a["lse"]),
                              a["B"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["chunk"], vp(a["ws"]), a["wsb"],
                              None)


def test_splitkv_argument_checks(L):
    assert _splitkv(L, Hq=6, Hkv=4) == 1
    assert _splitkv(L, chunk=1000) == 1       # not a multiple of the 64-key tile
    assert _splitkv(L, chunk=0) == 1
    assert _splitkv(L, S=0) == 1
    assert _splitkv(L, d=80) == 2
    assert _splitkv(L, s=0) == 1
    assert _splitkv(L, k=24) == 3
    assert _splitkv(L, ws=0) == 7
    need = L.attn_splitkv_workspace_size(2, 8, 2048, 128, 1024)
    assert need == 2 * 8 * 2 * 128 * 4 + 2 * 8 * 2 * 4
    assert _splitkv(L, wsb=need - 1) == 7
    assert L.attn_splitkv_workspace_size(2, 8, 2048, 128, 1000) == 0


def _paged(L, **kw):
    a = dict(q=16, k=16, v=16, bt=16, mb=8, ps=256, npg=64, s=16, o=16, lse=16, B=2, Hq=8, Hkv=2, d=128,
             scale=0.1, chunk=1024, ws=16, wsb=1 << 30)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd_splitkv_paged(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["bt"]), a["mb"], a["ps"], a["npg"],
                                    vp(a["s"]), vp(a["o"]), vp(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["d"],
                                    a["scale"], a["chunk"], vp(a["ws"]), a["wsb"], None)


def test_paged_splitkv_argument_checks(L):
    assert _paged(L, bt=0) == 1               # no block table
    assert _paged(L, ps=100) == 1             # page not a multiple of the 64-key tile
    assert _paged(L, ps=0) == 1
    assert _paged(L, mb=0) == 1
    assert _paged(L, npg=0) == 1
    assert _paged(L, ps=64, chunk=8192) == 2  # more pages per split than the kernel lists
    assert _paged(L, bt=18) == 3              # misaligned block table
    assert _paged(L, Hq=6, Hkv=4) == 1        # the checks of the contiguous call apply
    need = L.attn_splitkv_workspace_size(2, 8, 8 * 256, 128, 1024)   # capacity max_blocks * page_size
    assert _paged(L, wsb=need - 1) == 7


def _kvc(L, **kw):
    a = dict(q=16, k=16, v=16, s=16, S=512, o=16, lse=16, B=2, Hq=8, Hkv=2, Nq=40, d=128, causal=2, wl=-1, wr=-1,
             scale=0.1)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd_kvcache(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["s"]), a["S"], vp(a["o"]), vp(a["lse"]),
                              a["B"], a["Hq"], a["Hkv"], a["Nq"], a["d"], a["causal"], a["wl"], a["wr"],
                              a["scale"], None)


def test_kvcache_argument_checks(L):
    assert _kvc(L, causal=3) == 1
    assert _kvc(L, S=0) == 1
    assert _kvc(L, Hq=6, Hkv=4) == 1
    assert _kvc(L, s=0) == 1                  # no cache lengths
    assert _kvc(L, d=80) == 2
    assert _kvc(L, k=24) == 3
    assert _kvc(L, s=18) == 3                 # misaligned lengths
    assert _kvc(L, Nq=0) == 0                 # nothing to do


def _win(L, **kw):
    a = dict(q=16, k=16, v=16, o=16, lse=16, B=2, Hq=8, Hkv=2, Nq=300, Nk=300, d=128, causal=0, wl=127, wr=0,
             scale=0.1)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd_window(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["o"]), vp(a["lse"]), a["B"], a["Hq"],
                             a["Hkv"], a["Nq"], a["Nk"], a["d"], a["causal"], a["wl"], a["wr"], a["scale"], None)


def test_window_argument_checks(L):
    """Host checks run before anything is launched (no GPU needed): every
    window value is accepted (negative: unbounded side), the other checks
    are those of attn_fwd."""
    assert _win(L, causal=3) == 1
    assert _win(L, Hq=6, Hkv=4) == 1
    assert _win(L, d=96) == 2
    assert _win(L, q=0) == 1
    assert _win(L, k=8) == 3
    assert _win(L, scale=float("nan")) == 1
    assert _win(L, Nq=0) == 0
    assert _win(L, Nq=0, wl=-7, wr=1 << 30) == 0
    assert _win(L, Nq=(1 << 31) - 200, Nk=100) == 2   # Nq + Nk must leave room below 2^31
    assert _kvc(L, Nq=0, wl=5, wr=-3) == 0


def _noalloc(L, **kw):
    a = dict(q=16, k=16, v=16, s=16, S=2048, o=16, lse=16, B=2, Hq=8, Hkv=2, d=128, scale=0.1, chunk=1024)
    a.update(kw)
    vp = lambda x: ctypes.c_void_p(x) if x else None
    return L.attn_fwd_splitkv_noalloc(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["s"]), a["S"], vp(a["o"]),
                                      vp(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["d"], ctypes.c_float(a["scale"]),
                                      a["chunk"], None)


def test_noalloc_refuses_sizes_beyond_its_scratch(L):
    """The no-allocation decode checks its arguments with attn_fwd_splitkv's
    codes first, then refuses a problem whose partials exceed its fixed
    8 MiB scratch; every case here fails before any CUDA call (the pointers
    are never dereferenced)."""
    scratch_max = 8 << 20
    # 64 sequences x 32 heads x 32 splits x (128 + 1) floats: about 33 MB
    assert L.attn_splitkv_workspace_size(64, 32, 32768, 128, 1024) > scratch_max
    assert _noalloc(L, B=64, Hq=32, Hkv=8, S=32768) == 7          # ATTN_ERR_WORKSPACE
    # the other argument errors keep their own codes, also at sizes past the scratch
    assert _noalloc(L, B=64, Hq=32, Hkv=8, S=32768, d=256) == 2   # unsupported head dim
    assert _noalloc(L, B=64, Hq=32, Hkv=6, S=32768) == 1          # heads do not divide
    assert _noalloc(L, B=64, Hq=32, Hkv=8, S=32768, chunk=1000) == 1
    assert _noalloc(L, B=64, Hq=32, Hkv=8, S=32768, k=24) == 3    # misaligned
    assert _noalloc(L, B=64, Hq=32, Hkv=8, S=32768, s=0) == 1     # no cache lengths
    assert _noalloc(L, scale=float("nan")) == 1


def test_selftest_and_probe_argument_checks(L):
    """Host checks of the software-exp2 self-test and the read probe (no CUDA
    call is made for any of these)."""
    vp = ctypes.c_void_p
    assert L.attn_selftest_exp2_poly(None, None, 0, None) == 0          # nothing to do
    assert L.attn_selftest_exp2_poly(None, None, -1, None) == 1
    assert L.attn_selftest_exp2_poly(vp(16), None, 8, None) == 1
    assert L.attn_selftest_exp2_poly(vp(18), vp(16), 8, None) == 3      # not 4-byte aligned
    assert L.attn_probe_read_bandwidth(None, 0, None, None) == 0
    assert L.attn_probe_read_bandwidth(None, 64, vp(16), None) == 1
    assert L.attn_probe_read_bandwidth(vp(24), 64, vp(16), None) == 3   # buffer not 16-byte aligned
    assert L.attn_probe_read_bandwidth(vp(32), 40, vp(16), None) == 3   # size not a multiple of 16
    assert L.attn_probe_read_bandwidth(vp(32), 64, vp(12), None) == 3   # sink not 8-byte aligned
