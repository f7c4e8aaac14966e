"""C-ABI checks that need no GPU: the library builds, loads, exports exactly the
entry points include/fa2.h declares, and rejects bad arguments on the host
before any CUDA call.  (Compute calls are covered by the -m gpu tests.)"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from io_aware_exact_fa2_gb300 import build as fa2_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa2.h")

OK, INVALID, UNSUPPORTED, CUDA_ERR, TIMEOUT = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    path = fa2_build.build()
    from io_aware_exact_fa2_gb300 import _binding
    assert _binding.library_path() == path
    return _binding._lib


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa2_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert header_functions() == ["fa2_bwd", "fa2_bwd_ex", "fa2_bwd_window", "fa2_bwd_workspace_size", "fa2_fwd",
                                  "fa2_fwd_ex", "fa2_fwd_fp8",
                                  "fa2_fwd_from_host",
                                  "fa2_fwd_noalloc", "fa2_fwd_window", "fa2_fwd_ws", "fa2_get_device_error",
                                  "fa2_status_string", "fa2_version", "fa2_workspace_size"]


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


@pytest.mark.skipif(shutil.which("nm") is None, reason="binutils nm not available")
def test_library_exports_nothing_else(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa2_build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines()
                       if line.split() and line.split()[-2] in ("T", "W", "D", "B")})
    assert exported == header_functions()


def test_status_strings_and_version(lib):
    names = {OK: b"FA2_OK", INVALID: b"FA2_ERR_INVALID_ARG", UNSUPPORTED: b"FA2_ERR_UNSUPPORTED",
             CUDA_ERR: b"FA2_ERR_CUDA", TIMEOUT: b"FA2_ERR_TIMEOUT"}
    for code, name in names.items():
        assert lib.fa2_status_string(code) == name
    assert lib.fa2_status_string(99) == b"FA2_ERR_UNKNOWN"
    assert lib.fa2_version() == 100


# fake, never-dereferenced, 16-byte-aligned addresses: every case below must be
# rejected by host-side validation before the library makes any CUDA call
P = 0x10000


def call(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, Lq=8, Lk=8, D=64, causal=0, scale=0.125):
    return lib.fa2_fwd(q, k, v, o, lse, B, H, Lq, Lk, D, causal, scale, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=0), INVALID), (dict(k=0), INVALID), (dict(v=0), INVALID),
    (dict(o=0), INVALID), (dict(lse=0), INVALID),
    (dict(q=P + 8), INVALID), (dict(k=P + 2), INVALID), (dict(v=P + 4), INVALID),
    (dict(o=P + 1), INVALID), (dict(lse=P + 2), INVALID),
    (dict(B=0), INVALID), (dict(H=-1), INVALID), (dict(Lq=-1), INVALID),
    (dict(Lk=0), INVALID), (dict(D=0), INVALID),
    (dict(B=65536, H=65536), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-0.5), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(D=32), UNSUPPORTED), (dict(D=96), UNSUPPORTED), (dict(D=512), UNSUPPORTED),
    (dict(Lq=0), OK),
])
def test_host_validation(lib, kw, expect):
    assert call(lib, **kw) == expect


def test_from_host_validation(lib):
    args = [P] * 10
    f = lib.fa2_fwd_from_host
    bad = list(args)
    bad[0] = 0  # q_host
    assert f(*bad, 1, 1, 8, 8, 64, 0, 0.125, None) == INVALID
    bad = list(args)
    bad[6] = P + 8  # k_dev misaligned
    assert f(*bad, 1, 1, 8, 8, 64, 0, 0.125, None) == INVALID
    assert f(*args, 1, 1, 8, 8, 80, 0, 0.125, None) == UNSUPPORTED
    assert f(*args, 1, 1, 0, 8, 64, 0, 0.125, None) == OK


def test_workspace_entry_points_validation(lib):
    n = ctypes.c_size_t(123)
    f = lib.fa2_workspace_size
    assert f(1, 1, 8, 8, 64, 0, 0, None) == INVALID
    assert f(0, 1, 8, 8, 64, 0, 0, ctypes.byref(n)) == INVALID and n.value == 0
    assert f(1, 1, 8, 8, 96, 0, 0, ctypes.byref(n)) == UNSUPPORTED
    assert f(1, 1, 8, 8, 64, 1, 0, ctypes.byref(n)) == OK and n.value == 0   # causal: none needed
    assert f(1, 1, 0, 8, 64, 0, 0, ctypes.byref(n)) == OK and n.value == 0   # Lq == 0
    g = lib.fa2_fwd_ws
    args = [P] * 5 + [1, 1, 8, 8, 64, 0, 0.125]
    assert g(*args, P + 16, 1 << 20, None) == INVALID     # workspace not 256-byte aligned
    bad = list(args)
    bad[9] = 80
    assert g(*bad, P, 1 << 20, None) == UNSUPPORTED
    zero_q = list(args)
    zero_q[7] = 0
    assert g(*zero_q, 0, 0, None) == OK                   # Lq == 0 is a no-op


def test_no_gpu_reports_cuda_error_instead_of_crashing(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible; this checks the no-device path")
    assert call(lib) == CUDA_ERR


def test_binding_shape_checks():
    import torch
    from io_aware_exact_fa2_gb300 import _binding
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 9, 64, dtype=torch.bfloat16)
    o = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8, dtype=torch.float32)
    with pytest.raises(ValueError):
        _binding._check_shapes(q, k, k[:, :, :8], o, lse)
    with pytest.raises(TypeError):
        _binding._check_shapes(q.float(), k, k, o, lse)
    with pytest.raises(ValueError):
        _binding._check_shapes(q, k, k, o, lse[:, :, :7])
    assert _binding._check_shapes(q, k, k, o, lse) == (1, 2, 8, 9, 64)


def test_bwd_validation(lib):
    """Backward entry points reject bad arguments on the host, before any CUDA call."""
    n = ctypes.c_size_t(0)
    assert lib.fa2_bwd_workspace_size(2, 3, 100, 50, 128, ctypes.byref(n)) == OK
    assert n.value == 2 * 3 * 128 * 2 * 4   # (-lse2, -Delta) per row, 100 rows padded to 128
    assert lib.fa2_bwd_workspace_size(2, 3, 100, 50, 256, ctypes.byref(n)) == OK and n.value == 2 * 3 * 128 * 2 * 4
    assert lib.fa2_bwd_workspace_size(2, 3, 100, 50, 96, ctypes.byref(n)) == UNSUPPORTED
    assert lib.fa2_bwd_workspace_size(0, 3, 100, 50, 64, ctypes.byref(n)) == INVALID
    f = lib.fa2_bwd
    good = dict(q=P, k=P, v=P, o=P, lse=P, do=P, dq=P, dk=P, dv=P, B=1, H=1, Lq=8, Lk=8, D=64, causal=0,
                scale=0.125, ws=P, ws_bytes=4096)

    def call_bwd(**kw):
        a = dict(good, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["B"], a["H"],
                 a["Lq"], a["Lk"], a["D"], a["causal"], a["scale"], a["ws"], a["ws_bytes"], None)
    assert call_bwd(do=0) == INVALID
    assert call_bwd(dq=P + 8) == INVALID
    assert call_bwd(dk=0) == INVALID
    assert call_bwd(ws=0) == INVALID
    assert call_bwd(ws_bytes=4) == INVALID
    assert call_bwd(D=96) == UNSUPPORTED
    assert call_bwd(scale=float("nan")) == INVALID


def test_bwd_window_validation(lib):
    """fa2_bwd_window: a negative window and Lq > Lk are rejected before any CUDA call, and
    otherwise it checks its arguments as fa2_bwd does."""
    f = lib.fa2_bwd_window

    def call(Lq=8, Lk=8, D=64, window=4, do=P, ws_bytes=4096):
        return f(P, P, P, P, P, do, P, P, P, 1, 1, Lq, Lk, D, window, 0.125, P, ws_bytes, None)
    assert call(window=-1) == INVALID
    assert call(Lq=9) == INVALID
    assert call(do=0) == INVALID
    assert call(ws_bytes=4) == INVALID
    assert call(D=96) == UNSUPPORTED


def test_bwd_ex_validation(lib):
    """fa2_bwd_ex rejects strides that are not positive multiples of 8 elements (or above
    2^38) and a bad window, before any CUDA call."""
    f = lib.fa2_bwd_ex
    ll3 = ctypes.c_longlong * 3

    def call(bad=None, at=0, causal=1, window=-1, Lq=8, Lk=8):
        arrays = [None] * 8
        if bad is not None:
            arrays[at] = ll3(*bad)
        return f(P, P, P, P, P, P, P, P, P, 1, 1, Lq, Lk, 64, *arrays, causal, window, 0.125, P, 4096, None)
    for at in range(8):
        assert call((8 * 64, 64, 68), at) == INVALID     # row stride not a multiple of 8
        assert call((8 * 64, 0, 64), at) == INVALID      # zero head stride
        assert call((1 << 39, 512, 64), at) == INVALID   # beyond 2^38
    assert call(window=-2) == INVALID
    assert call(window=4, causal=0) == INVALID
    assert call(window=4, Lq=9) == INVALID


def test_window_validation(lib):
    """fa2_fwd_window rejects a negative window and Lq > Lk before any CUDA call."""
    f = lib.fa2_fwd_window
    assert f(P, P, P, P, P, 1, 1, 8, 8, 64, -1, 0.125, None) == INVALID
    assert f(P, P, P, P, P, 1, 1, 9, 8, 64, 4, 0.125, None) == INVALID
    assert f(0, P, P, P, P, 1, 1, 8, 8, 64, 4, 0.125, None) == INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 8, 96, 4, 0.125, None) == UNSUPPORTED
    assert f(P, P, P, P, P, 1, 1, 0, 8, 64, 4, 0.125, None) == OK   # Lq == 0: no-op


def test_fwd_ex_validation(lib):
    """fa2_fwd_ex rejects bad strides, windows and workspaces before any CUDA call."""
    f = lib.fa2_fwd_ex
    L3 = ctypes.c_longlong * 3

    def call(qs=None, ks=None, vs=None, os_=None, causal=0, window=-1, ws=None, Lq=8, Lk=8, D=64):
        arr = [None if s is None else L3(*s) for s in (qs, ks, vs, os_)]
        return f(P, P, P, P, P, 1, 2, Lq, Lk, D, *arr, causal, window, 0.125, ws, 0, None)

    assert call(Lq=0) == OK                                       # contiguous, Lq == 0: no-op
    assert call(qs=(2 * 8 * 64, 64, 2 * 64), Lq=0) == OK          # a [B, L, H, D] view of q
    assert call(qs=(1024, 64, 12)) == INVALID                     # row stride not a multiple of 8
    assert call(ks=(1024, 0, 64)) == INVALID                      # zero stride
    assert call(vs=(-1024, 512, 64)) == INVALID                   # negative stride
    assert call(os_=(1 << 39, 512, 64)) == INVALID                # beyond what a TMA map can address
    assert call(window=-2) == INVALID
    assert call(window=4) == INVALID                              # a window needs causal
    assert call(causal=1, window=4, Lq=9, Lk=8) == INVALID        # and Lq <= Lk
    assert call(ws=P + 16) == INVALID                             # workspace not 256-byte aligned
    assert call(D=96) == UNSUPPORTED


def test_fwd_fp8_validation(lib):
    """fa2_fwd_fp8's host-side checks (no CUDA call is made for these): the descales are
    required and 4-byte aligned, D must be 128, Lq == 0 is a no-op."""
    P = 0x10000
    f = lib.fa2_fwd_fp8
    # q, k, v, dq, dk, dv, o, lse, B, H, Lq, Lk, D, causal, scale, ws, ws_bytes, stream
    assert f(P, P, P, None, P, P, P, P, 1, 1, 8, 8, 128, 0, 0.1, None, 0, None) == INVALID
    assert f(P, P, P, P, P + 2, P, P, P, 1, 1, 8, 8, 128, 0, 0.1, None, 0, None) == INVALID
    assert f(P, P, P, P, P, None, P, P, 1, 1, 8, 8, 128, 0, 0.1, None, 0, None) == INVALID
    assert f(P, P, P, P, P, P, P, P, 1, 1, 8, 8, 64, 0, 0.1, None, 0, None) == UNSUPPORTED
    assert f(P, P, P, P, P, P, P, P, 1, 1, 8, 8, 96, 0, 0.1, None, 0, None) == UNSUPPORTED
    assert f(P, P, P, P, P, P, P + 8, P, 1, 1, 8, 8, 128, 0, 0.1, None, 0, None) == INVALID   # o misaligned
    assert f(P, P, P, P, P, P, P, P, 1, 1, 0, 8, 128, 0, 0.1, None, 0, None) == OK   # Lq == 0
    assert f(P, P, P, P, P, P, P, P, 1, 1, 8, 8, 128, 0, float("nan"), None, 0, None) == INVALID
