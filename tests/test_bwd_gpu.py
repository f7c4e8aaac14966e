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


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_c1_every_element(D, causal):
    inputs, got = run_bwd(1, 2, 128, 128, D, causal, seed=5100 + D)
    compare_grads(inputs, got, causal)


@pytest.mark.parametrize("D", [64, 128, 256])
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


@pytest.mark.parametrize("D", [128, 256])
def test_deterministic(D):
    """No atomics: the same inputs give bit-identical gradients."""
    _, a = run_bwd(2, 2, 333, 400, D, True, seed=5600)
    _, b = run_bwd(2, 2, 333, 400, D, True, seed=5600)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def delta_term(q, k, v, do, o_stored, scale, heads, ref=None, o_exact=None):
    """Relative rms, per gradient, of the error that Delta = rowsum(dO * O) takes from the
    STORED (bf16) O ("Chapter 08: Flash Attention -- blocked attention", section 6.2
    defines Delta from the forward's output): dDelta_i = sum_d dO_id (O~_id - O_id), and
    dS = P (dP - Delta) passes -P dDelta on, so dQ errs by -scale dDelta (P K) and dK by
    -scale (P dDelta)^T Q.  Where one key dominates a row, dP - Delta cancels and this
    term is no longer small next to the bf16 operand rounding."""
    import oracle as orc
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    # the oracle's gradients of these heads (only their rms is used) and its exact O, unless given
    dq, dk = ref[:2] if ref is not None else orc.gradients(q, k, v, do, False, scale, heads=heads)[:2]
    if o_exact is None:
        o_exact, _ = orc.attention(q, k, v, False, scale)
    out = ("dq", "dk")
    Q, K, DO = (t.double().numpy().reshape(B * H, -1, D)[heads] for t in (q, k, do))
    OE = o_exact.reshape(B * H, Lq, D)[heads]
    OS = o_stored.double().numpy().reshape(B * H, Lq, D)[heads]
    num = {"dq": 0.0, "dk": 0.0}
    den = {"dq": 0.0, "dk": 0.0}
    ref = {"dq": dq, "dk": dk}
    for n in range(len(heads)):
        s = scale * Q[n] @ K[n].T
        P = np.exp(s - s.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        dd = (DO[n] * (OS[n] - OE[n])).sum(1)
        e = {"dq": scale * dd[:, None] * (P @ K[n]), "dk": scale * (P * dd[:, None]).T @ Q[n]}
        for g in out:
            num[g] += np.sum(e[g] ** 2)
            den[g] += np.sum(ref[g][n] ** 2)
    return {g: float(np.sqrt(num[g] / den[g])) for g in out}


def test_d256_peaky_workload_shape_sampled_heads():
    """B2 H8 Lq2000 Lk3000 D256 with every 64th key row x8 (the peaky D = 256 workload):
    every element of two heads.  At D = 256 two CTAs share each resident tile, each
    accumulating one half of the gradient columns.

    Tolerance: the module's bar is twice the bf16 operand/output rounding predicted for
    N(0, 1) rows (~2.5e-3 rel rms).  Here each row has a dominant key, so the rounding
    of the stored O inside Delta adds an error of its own (delta_term: about 4.5e-3 rel
    rms for dq and dk on these heads, computed from the exact and stored O).  The bar
    for dq and dk is twice the two combined, sqrt(2.5e-3^2 + term^2); dv (no Delta in
    it) keeps the module's bar."""
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_fwd, fa2_get_device_error
    from io_aware_exact_fa2_gb300.workloads import WORKLOADS, workload_inputs
    w = WORKLOADS["c5"]
    dev = torch.device("cuda:0")
    q, k, v = workload_inputs(w)
    do = make_qkv(w.B, w.H, w.Lq, w.Lq, w.D, seed_base=w.seed_base + 7)[0]
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty(w.B, w.H, w.Lq, w.D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, w.Lq, dtype=torch.float32, device=dev)
    fa2_fwd(qd, kd, vd, o, lse, False, w.scale)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    fa2_bwd(qd, kd, vd, o, lse, dod, *grads, False, w.scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    heads = [0, 15]
    term = delta_term(q, k, v, do, o.cpu(), w.scale, heads)
    ref = oracle.gradients(q, k, v, do, False, w.scale, heads=heads)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref[:3]):
        g = g.cpu().double().reshape(w.B * w.H, *g.shape[2:]).numpy()[heads]
        assert np.isfinite(g).all(), name
        err = np.abs(g - r)
        rel_rms = np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(r ** 2))
        rel_max = err.max() / np.abs(r).max()
        bar = 2 * np.hypot(2.5e-3, term[name]) if name in term else REL_RMS
        print(f"c5 backward {name}: rel rms {rel_rms:.2e} (bar {bar:.2e}), rel max {rel_max:.2e}")
        assert rel_rms <= bar, (name, rel_rms, bar)
        assert rel_max <= REL_MAX, (name, rel_max)


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
    t = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 8, device=dev)
    with pytest.raises(Fa2Error):
        fa2_bwd(t, t, t, t, lse, t, torch.empty_like(t), torch.empty_like(t), torch.empty_like(t), False)
