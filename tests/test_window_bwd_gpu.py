"""Backward pass of the causal sliding window ("Flash Attention: principles and
implementation", section 6.3: window_size = (w, 0) with causal) on the GPU against
the oracle's window gradients.  Those are the definition of "Chapter 08: Flash
Attention -- blocked attention", section 6, under the window's mask, and they are
pinned by finite differences of the window forward.

The tolerance is the one of the plain backward, for the same reasons (bf16
outputs; P and dS as bf16 MMA operands): per tensor rms(err)/rms(ref) <= 5e-3 and
max|err| <= 1e-2 * max|ref|.  For tensors that are zero in exact arithmetic the
bars apply to the absolute error instead.  With w = 0 each query sees only its own
key, so P = 1, dS = 0, dq = dk = 0 and dv = dO."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL_RMS = 5e-3
REL_MAX = 1e-2


def run(B, H, Lq, Lk, D, window, seed):
    from io_aware_exact_fa2_gb300 import fa2_bwd_window, fa2_fwd_window, fa2_get_device_error
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=seed)
    do = make_qkv(B, H, Lq, Lq, D, seed_base=seed + 500)[0]
    scale = D ** -0.5
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device=DEV)
    fa2_fwd_window(qd, kd, vd, o, lse, window, scale)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    fa2_bwd_window(qd, kd, vd, o, lse, dod, *grads, window, scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    return (q, k, v, do, scale), [g.cpu() for g in grads]


def check(inputs, got, window, heads=None):
    q, k, v, do, scale = inputs
    B, H = q.shape[:2]
    ref = oracle.gradients(q, k, v, do, True, scale, heads=heads, window=window)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref[:3]):
        g = g.double().reshape(B * H, *g.shape[2:]).numpy()
        if heads is not None:
            g = g[heads]
        else:
            r = r.reshape(g.shape)
        assert np.isfinite(g).all(), name
        err = np.abs(g - r)
        rms_ref, max_ref = np.sqrt(np.mean(r ** 2)), np.abs(r).max()
        rms_err = np.sqrt(np.mean(err ** 2))
        assert rms_err <= REL_RMS * (rms_ref if rms_ref > 1e-6 else 1.0), (name, rms_err, rms_ref)
        assert err.max() <= REL_MAX * (max_ref if max_ref > 1e-6 else 1.0), (name, err.max(), max_ref)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("window", [0, 1, 63, 100, 200])
def test_window_backward_every_element(D, window):
    """Ragged Lq < Lk: band edges inside and across the 64-row tiles of both kernels."""
    inputs, got = run(1, 2, 300, 457, D, window, seed=7100 + window + D)
    check(inputs, got, window)
    # keys no query sees (j >= Lq) get zero gradients
    assert torch.count_nonzero(got[1][:, :, 300:]) == 0 and torch.count_nonzero(got[2][:, :, 300:]) == 0


def test_zero_window_is_the_diagonal():
    """w = 0: P = 1 on the diagonal, so dS = 0 and dv = dO (the bf16 dO itself)."""
    inputs, got = run(1, 2, 200, 200, 64, 0, seed=7300)
    do = inputs[3]
    assert torch.equal(got[2], do)
    assert float(got[0].abs().max()) <= 1e-2 and float(got[1].abs().max()) <= 1e-2


@pytest.mark.parametrize("D", [64, 128])
def test_wide_window_is_plain_causal(D):
    """A window covering every earlier key gives the plain causal backward bit for bit."""
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_fwd
    B, H, L = 1, 3, 333
    inputs, got = run(B, H, L, L, D, L, seed=7400 + D)
    q, k, v, do, scale = inputs
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o = torch.empty(B, H, L, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, L, dtype=torch.float32, device=DEV)
    fa2_fwd(qd, kd, vd, o, lse, True, scale)
    ref = [torch.empty_like(t) for t in (qd, kd, vd)]
    fa2_bwd(qd, kd, vd, o, lse, dod, *ref, True, scale)
    for g, r in zip(got, ref):
        assert torch.equal(g, r.cpu())


def test_window_backward_multi_tile_heads():
    """A longer sequence, many query and key tiles per head, checked on sampled heads."""
    inputs, got = run(2, 4, 2048, 2048, 128, 256, seed=7500)
    check(inputs, got, 256, heads=[0, 5])
