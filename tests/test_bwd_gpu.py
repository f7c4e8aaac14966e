"""Backward pass (Chapter 08: Flash Attention -- blocked attention, section 6)
on the GPU against the fp64 oracle's gradients.

Tolerance, from the arithmetic: dq, dk, dv are stored as bf16 (relative
rounding up to 2^-9, rms ~1.1e-3 of the value), and P and dS enter the
gradient MMAs as bf16 operands (the same relative rounding per term, fp32
accumulation).  Together they give a relative rms error of ~2-3e-3 and a
largest error of ~5e-3 of the tensor's largest magnitude; the bar is twice
that: rms(err)/rms(ref) <= 5e-3 and max|err| <= 1e-2 * max|ref|, per tensor."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

REL_RMS = 5e-3
REL_MAX = 1e-2


def run_bwd(B, H, Lq, Lk, D, causal, seed, dout_scale=1.0):
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_fwd, fa2_get_device_error
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=seed)
    do = make_qkv(B, H, Lq, Lq, D, seed_base=seed + 500)[0]
    if dout_scale != 1.0:
        do = (do.float() * dout_scale).to(torch.bfloat16)
    scale = D ** -0.5
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
    fa2_fwd(qd, kd, vd, o, lse, causal, scale)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    fa2_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, causal, scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    return (q, k, v, do, scale), (dq.cpu(), dk.cpu(), dv.cpu())


def compare_grads(inputs, got, causal, heads=None):
    q, k, v, do, scale = inputs
    B, H = q.shape[:2]
    ref = oracle.gradients(q, k, v, do, causal, scale, heads=heads)
    report = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref[:3]):
        g = g.double().reshape(B * H, *g.shape[2:]).numpy()
        if heads is not None:
            g = g[heads]
        else:
            r = r.reshape(g.shape)
        assert np.isfinite(g).all(), name
        err = np.abs(g - r)
        rms_ref = np.sqrt(np.mean(r ** 2))
        rel_rms = np.sqrt(np.mean(err ** 2)) / rms_ref if rms_ref > 0 else float(np.sqrt(np.mean(err ** 2)))
        rel_max = err.max() / np.abs(r).max() if np.abs(r).max() > 0 else float(err.max())
        report[name] = (rel_rms, rel_max)
        assert rel_rms <= REL_RMS, (name, rel_rms)
        assert rel_max <= REL_MAX, (name, rel_max)
    return report


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_c1_every_element(D, causal):
    inputs, got = run_bwd(1, 2, 128, 128, D, causal, seed=5100 + D)
    compare_grads(inputs, got, causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_ragged_multi_tile(D, causal):
    """Lq, Lk not multiples of any tile (query tiles of 64 and 128, key tiles of 64 and 128)."""
    inputs, got = run_bwd(2, 3, 300, 457, D, causal, seed=5200 + D)
    compare_grads(inputs, got, causal)


@pytest.mark.parametrize("Lq,Lk", [(457, 300), (200, 600), (129, 1), (1, 77)])
def test_causal_unequal_lengths(Lq, Lk):
    """Top-left causal rule with Lq != Lk: keys no query sees get zero gradients."""
    inputs, got = run_bwd(1, 2, Lq, Lk, 128, True, seed=5300 + Lq)
    compare_grads(inputs, got, True)
    if Lk > Lq:
        assert torch.count_nonzero(got[1][:, :, Lq:]) == 0 and torch.count_nonzero(got[2][:, :, Lq:]) == 0


@pytest.mark.parametrize("D,causal", [(64, True), (64, False), (128, True)], ids=["d64-causal", "d64-noncausal", "d128-causal"])
def test_more_key_tiles_than_sms(D, causal):
    """More key tiles (5 per head x 64 heads) than SMs, so the dK/dV grid runs in
    several waves; when causal with Lk > Lq, tiles no query sees (zero gradients, no
    MMAs) sit between tiles with steps in every wave."""
    Lq, Lk = 200, 600
    inputs, got = run_bwd(1, 64, Lq, Lk, D, causal, seed=5600 + D)
    compare_grads(inputs, got, causal, heads=[0, 17, 38, 63])
    if causal:
        assert torch.count_nonzero(got[1][:, :, Lq:]) == 0 and torch.count_nonzero(got[2][:, :, Lq:]) == 0


def test_many_heads_and_large_dout():
    """More CTAs than SMs in both kernels, and a dO of larger magnitude (x16, exact in bf16)."""
    inputs, got = run_bwd(4, 16, 320, 320, 64, False, seed=5400, dout_scale=16.0)
    compare_grads(inputs, got, False, heads=[0, 17, 63])


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_c3_size_sampled_heads(causal):
    """The forward bench's shape (B2 H16 L4096 D128): every element of two heads."""
    inputs, got = run_bwd(2, 16, 4096, 4096, 128, causal, seed=5500)
    compare_grads(inputs, got, causal, heads=[0, 31])


def test_deterministic():
    """No atomics: the same inputs give bit-identical gradients."""
    _, a = run_bwd(2, 2, 333, 400, 128, True, seed=5600)
    _, b = run_bwd(2, 2, 333, 400, 128, True, seed=5600)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_no_queries_zero_key_gradients():
    """Lq == 0: no query sees any key, so dk and dv are zeroed (and nothing else is
    touched); the query-side buffers are never read."""
    from io_aware_exact_fa2_gb300 import _binding
    dev = torch.device("cuda:0")
    B, H, Lk, D = 1, 2, 50, 64
    k = torch.randn(B, H, Lk, D, device=dev).to(torch.bfloat16)
    v = torch.randn(B, H, Lk, D, device=dev).to(torch.bfloat16)
    dummy = torch.zeros(64, dtype=torch.bfloat16, device=dev)   # stands in for the empty q-side tensors
    lse = torch.zeros(4, dtype=torch.float32, device=dev)
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    p = dummy.data_ptr()
    st = _binding._lib.fa2_bwd(p, k.data_ptr(), v.data_ptr(), p, lse.data_ptr(), p, p, dk.data_ptr(), dv.data_ptr(),
                               B, H, 0, Lk, D, 0, 0.125, None, 0, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0
    assert torch.count_nonzero(dummy) == 0


def test_unsupported_head_dim():
    from io_aware_exact_fa2_gb300 import Fa2Error, fa2_bwd
    dev = torch.device("cuda:0")
    t = torch.zeros(1, 1, 8, 256, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 8, device=dev)
    with pytest.raises(Fa2Error):
        fa2_bwd(t, t, t, t, lse, t, torch.empty_like(t), torch.empty_like(t), torch.empty_like(t), False)
