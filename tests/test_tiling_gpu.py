"""Tiling independence: builds of the library with other tile configurations
(one or two Q tiles per CTA, one or two warps per softmax row, other ring
depths) compute the same attention -- each is checked against the fp64 oracle
on ragged causal and non-causal shapes.  The result of the method does not
depend on how the score matrix is blocked."""
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
    "d128_nq1_cs1": (128, ["-DFA2_D128_NQ=1"]),
    "d128_nq1_cs2": (128, ["-DFA2_D128_NQ=1", "-DFA2_D128_CS=2"]),
    "d128_nq2_cs2": (128, ["-DFA2_D128_CS=2"]),
    "d256_cs2": (256, ["-DFA2_D256_CS=2"]),
}


@pytest.fixture(scope="module")
def variant_libs(tmp_path_factory):
    libs = {}
    for name, (_, flags) in VARIANTS.items():
        d = tmp_path_factory.mktemp(name)
        path = fa2_build.build(extra_flags=flags, lib_path=str(d / "lib.so"), build_dir=str(d))
        lib = ctypes.CDLL(path)
        lib.fa2_fwd.restype = ctypes.c_int
        lib.fa2_fwd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_void_p]
        lib.fa2_get_device_error.restype = ctypes.c_int
        lib.fa2_get_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
        libs[name] = lib
    return libs


@pytest.mark.parametrize("name", list(VARIANTS))
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_variant_matches_oracle(variant_libs, name, causal):
    D = VARIANTS[name][0]
    lib = variant_libs[name]
    B, H, Lq, Lk = 2, 2, 333, 517
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=1200 + D)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=dev)
    st = lib.fa2_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     B, H, Lq, Lk, D, int(causal), scale_of(D), None)
    assert st == 0
    detail = ctypes.c_int(0)
    assert lib.fa2_get_device_error(None, ctypes.byref(detail)) == 0, detail.value
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale_of(D))
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref)
