"""Tiling independence: builds of the library with other tile configurations
(one or two Q tiles per CTA, one or two warps per softmax row, other ring
depths, Q kept in TMEM or in shared memory) compute the same attention -- each
is checked against the fp64 oracle on ragged causal and non-causal shapes, with
whole work units and with the split schedule.  The result of the method does
not depend on how the score matrix is blocked."""
import ctypes

import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300 import build as fa2_build
from io_aware_exact_fa2_gb300.workloads import make_qkv
from parity import compare, scale_of

pytestmark = pytest.mark.gpu

VARIANTS = {
    "d64_nq1_cs2_ks4": (64, ["-DFA2_D64_NQ=1", "-DFA2_D64_KS=4", "-DFA2_D64_CS=2"]),
    "d128_nq1_cs2": (128, ["-DFA2_D128_NQ=1", "-DFA2_D128_CS=2"]),
    # Q kept in TMEM (two buffers at D = 128, one at D = 256, which is that size's default)
    "d128_nq1_qt": (128, ["-DFA2_D128_NQ=1", "-DFA2_D128_QT=1"]),
    "d128_nq1_cs2_qt": (128, ["-DFA2_D128_NQ=1", "-DFA2_D128_CS=2", "-DFA2_D128_QT=1"]),
    "d256_q_in_smem": (256, ["-DFA2_D256_QT=0"]),
}

# (B, H, Lq, Lk): ragged tiles, and more work units than SMs so that CTAs move on
# from one unit to the next (Q buffers and barrier phases carried across units)
SHAPES = {"ragged": (2, 2, 333, 517), "many_units": (4, 20, 300, 257)}


@pytest.fixture(scope="module")
def variant_libs(tmp_path_factory):
    libs = {}
    for name, (_, flags) in VARIANTS.items():
        d = tmp_path_factory.mktemp(name)
        path = fa2_build.build(extra_flags=flags, lib_path=str(d / "lib.so"), build_dir=str(d))
        lib = ctypes.CDLL(path)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.fa2_fwd.restype = i32
        lib.fa2_fwd.argtypes = [vp] * 5 + [i32] * 6 + [ctypes.c_float, vp]
        lib.fa2_fwd_ws.restype = i32
        lib.fa2_fwd_ws.argtypes = [vp] * 5 + [i32] * 6 + [ctypes.c_float, vp, ctypes.c_size_t, vp]
        lib.fa2_workspace_size.restype = i32
        lib.fa2_workspace_size.argtypes = [i32] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
        lib.fa2_get_device_error.restype = i32
        lib.fa2_get_device_error.argtypes = [vp, ctypes.POINTER(i32)]
        libs[name] = lib
    return libs


@pytest.mark.parametrize("name", list(VARIANTS))
@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("mode", ["noncausal", "causal", "noncausal_split"])
def test_variant_matches_oracle(variant_libs, name, shape, mode, monkeypatch):
    D = VARIANTS[name][0]
    lib = variant_libs[name]
    B, H, Lq, Lk = SHAPES[shape]
    causal = mode == "causal"
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=1200 + D + Lq)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=dev)
    args = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
            B, H, Lq, Lk, D, int(causal), scale_of(D))
    if mode == "noncausal_split":
        monkeypatch.setenv("FA2_SPLIT", "always")
        n = ctypes.c_size_t(0)
        assert lib.fa2_workspace_size(B, H, Lq, Lk, D, 0, 0, ctypes.byref(n)) == 0 and n.value > 0
        ws = torch.zeros(n.value, dtype=torch.uint8, device=dev)
        st = lib.fa2_fwd_ws(*args, ws.data_ptr(), n.value, None)
    else:
        st = lib.fa2_fwd(*args, None)
    assert st == 0
    detail = ctypes.c_int(0)
    assert lib.fa2_get_device_error(None, ctypes.byref(detail)) == 0, detail.value
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale_of(D))
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref)
    if mode == "noncausal_split":
        assert torch.count_nonzero(ws[:256]) == 0
