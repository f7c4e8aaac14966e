"""Pins of the oracle's backward pass (Chapter 08: Flash Attention -- blocked
attention, section 6), each against something other than its own formulas:

- central finite differences of the oracle's own forward definition (the
  gradient of L = sum(dO * O) with respect to every input element);
- torch autograd in fp64 on an explicitly materialised softmax (a library
  cross-check that shares no code with the oracle);
- exact invariants: rows of P sum to one (so sum_j dV_j = sum_i dO_i), rows of
  dS sum to zero (so sum_j dK_j = 0), a constant added to every value row
  changes neither dQ nor dK nor dV, gradients are linear in dO, and causal row 0
  (which sees only key 0) has dQ = 0;
- a closed form: with Q = 0 every visible key gets weight 1/|A_i|.
"""
import numpy as np
import pytest
import torch

import oracle


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def loss(q, k, v, do, causal, scale):
    o, _ = oracle.forward_f64(q, k, v, causal, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
@pytest.mark.parametrize("Lq,Lk", [(5, 5), (4, 7), (6, 3)])
def test_gradients_match_finite_differences(causal, Lq, Lk):
    B, H, D, scale = 1, 2, 3, 0.8
    q, k, v, do = rand((B, H, Lq, D), 1), rand((B, H, Lk, D), 2), rand((B, H, Lk, D), 3), rand((B, H, Lq, D), 4)
    dq, dk, dv, _ = oracle.gradients_f64(q, k, v, do, causal, scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = loss(*[xp if n == name else args[n] for n in ("q", "k", "v")], do, causal, scale)
            lm = loss(*[xm if n == name else args[n] for n in ("q", "k", "v")], do, causal, scale)
            num[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(num - g)) < 2e-7, (name, np.max(np.abs(num - g)))


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_gradients_match_torch_autograd(causal):
    B, H, Lq, Lk, D, scale = 2, 3, 9, 11, 4, 0.35
    q, k, v, do = rand((B, H, Lq, D), 5), rand((B, H, Lk, D), 6), rand((B, H, Lk, D), 7), rand((B, H, Lq, D), 8)
    dq, dk, dv, delta = oracle.gradients_f64(q, k, v, do, causal, scale)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = scale * qt @ kt.transpose(-1, -2)
    if causal:
        keep = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None]
        s = s.masked_fill(~keep, float("-inf"))
    o = torch.softmax(s, dim=-1) @ vt
    (o * torch.tensor(do)).sum().backward()
    for got, want in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.max(np.abs(got - want.numpy())) < 1e-12
    assert np.max(np.abs(delta - np.sum(do * o.detach().numpy(), axis=-1))) < 1e-12


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_gradient_invariants(causal):
    B, H, Lq, Lk, D, scale = 1, 2, 12, 12, 5, 0.5
    q, k, v, do = rand((B, H, Lq, D), 9), rand((B, H, Lk, D), 10), rand((B, H, Lk, D), 11), rand((B, H, Lq, D), 12)
    dq, dk, dv, _ = oracle.gradients_f64(q, k, v, do, causal, scale)
    # rows of P sum to one: the value gradient collects every row's dO once
    assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) < 1e-12
    # rows of dS sum to zero: the key gradients cancel
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12
    # a constant added to every value row leaves all gradients unchanged
    shift = rand((1, 1, 1, D), 13)
    dq2, dk2, dv2, _ = oracle.gradients_f64(q, k, v + shift, do, causal, scale)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        assert np.max(np.abs(a - b)) < 1e-12
    # linear in dO
    dq3, dk3, dv3, _ = oracle.gradients_f64(q, k, v, 2.0 * do, causal, scale)
    for a, b in ((dq, dq3), (dk, dk3), (dv, dv3)):
        assert np.array_equal(2.0 * a, b)
    if causal:
        # row 0 sees only key 0: P = 1, dS = dO.(V0 - O0) = 0
        assert np.max(np.abs(dq[:, :, 0])) < 1e-15


def test_uniform_scores_closed_form():
    """Q = 0: every key gets weight 1/Lk, so dV_j = mean over rows of dO and
    dQ_i = (scale/Lk) sum_j (dO_i . (V_j - mean V)) K_j."""
    B, H, Lq, Lk, D, scale = 1, 1, 6, 8, 3, 0.9
    q = np.zeros((B, H, Lq, D))
    k, v, do = rand((B, H, Lk, D), 14), rand((B, H, Lk, D), 15), rand((B, H, Lq, D), 16)
    dq, dk, dv, _ = oracle.gradients_f64(q, k, v, do, False, scale)
    want_dv = np.broadcast_to(do.sum(axis=2, keepdims=True) / Lk, dv.shape)
    assert np.max(np.abs(dv - want_dv)) < 1e-14
    vbar = v.mean(axis=2, keepdims=True)
    w = np.einsum("bhid,bhjd->bhij", do, v - vbar)          # dO_i . (V_j - mean V)
    want_dq = scale / Lk * np.einsum("bhij,bhjd->bhid", w, k)
    assert np.max(np.abs(dq - want_dq)) < 1e-13
    # and dK_j = (scale/Lk) sum_i w_ij Q_i = 0 with Q = 0
    assert np.max(np.abs(dk)) == 0.0


def test_bf16_wrapper_widens_exactly_and_selects_heads():
    """gradients() on bf16 tensors equals gradients_f64() on their exact fp64 values,
    for all heads and for a selection of heads."""
    from io_aware_exact_fa2_gb300.workloads import make_qkv
    q, k, v = make_qkv(2, 2, 7, 9, 8, seed_base=77)
    do = make_qkv(2, 2, 7, 7, 8, seed_base=78)[0]
    full = oracle.gradients(q, k, v, do, True, 0.4)
    ref = oracle.gradients_f64(*(t.double().numpy() for t in (q, k, v, do)), True, 0.4)
    for a, b in zip(full, ref):
        assert np.array_equal(a, b)
    part = oracle.gradients(q, k, v, do, True, 0.4, heads=[3, 1])
    for a, b in zip(part, full):
        flat = b.reshape(4, *b.shape[2:])
        assert np.array_equal(a, flat[[3, 1]])
