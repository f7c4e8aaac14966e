"""Pins of the oracle's sliding-window attention ("Flash Attention: principles and
implementation", section 6.3: window_size = (w, 0) with causal -- query i sees keys
i - w <= j <= i), each against something other than the oracle's own mask:

- a window covering every earlier key is plain causal attention (same result);
- w = 0 leaves one key per row: O_i = V_i and LSE_i = s_ii exactly;
- torch fp64 softmax with an explicitly built band mask (a library cross-check);
- rows never see keys outside their band: changing those keys changes nothing;
- the window's gradients match finite differences of the window forward.
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv


def test_wide_window_is_causal():
    q, k, v = make_qkv(2, 2, 40, 40, 16, seed_base=8100)
    for w in (39, 40, 1000):
        o_w, l_w = oracle.attention(q, k, v, True, 0.25, window=w)
        o_c, l_c = oracle.attention(q, k, v, True, 0.25)
        assert np.array_equal(o_w, o_c) and np.array_equal(l_w, l_c)


def test_zero_window_keeps_the_diagonal_only():
    q, k, v = make_qkv(1, 2, 9, 12, 8, seed_base=8200)
    o, lse = oracle.attention(q, k, v, True, 0.5, window=0)
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    assert np.array_equal(o, vf[:, :, :9])
    s_ii = 0.5 * np.einsum("bhid,bhid->bhi", qf, kf[:, :, :9])
    assert np.max(np.abs(lse - s_ii)) < 1e-14


@pytest.mark.parametrize("w", [1, 3, 7])
def test_band_matches_torch_masked_softmax(w):
    B, H, Lq, Lk, D, scale = 2, 2, 13, 17, 8, 0.3
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=8300 + w)
    o, lse = oracle.attention(q, k, v, True, scale, window=w)
    qf, kf, vf = (t.double() for t in (q, k, v))
    s = scale * qf @ kf.transpose(-1, -2)
    i = torch.arange(Lq)[:, None]
    j = torch.arange(Lk)[None, :]
    s = s.masked_fill(~((j <= i) & (j >= i - w)), float("-inf"))
    assert np.max(np.abs(o - (torch.softmax(s, -1) @ vf).numpy())) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(s, -1).numpy())) < 1e-12


def test_keys_outside_the_band_do_not_matter():
    w = 4
    q, k, v = make_qkv(1, 1, 20, 20, 8, seed_base=8400)
    o, lse = oracle.attention(q, k, v, True, 0.4, window=w)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, :3] = 7.0       # keys 0..2 are outside every band of rows i >= w + 3
    v2[:, :, :3] = -5.0
    o2, lse2 = oracle.attention(q, k2, v2, True, 0.4, window=w)
    assert np.array_equal(o[:, :, w + 3:], o2[:, :, w + 3:])
    assert np.array_equal(lse[:, :, w + 3:], lse2[:, :, w + 3:])
    assert not np.array_equal(o[:, :, :w + 3], o2[:, :, :w + 3])


def test_window_gradients_match_finite_differences():
    rng = np.random.default_rng(8500)
    B, H, Lq, Lk, D, scale, w = 1, 1, 6, 7, 3, 0.7, 2
    q, k, v, do = (rng.standard_normal(s) for s in ((B, H, Lq, D), (B, H, Lk, D), (B, H, Lk, D), (B, H, Lq, D)))
    dq, dk, dv, _ = oracle.gradients_f64(q, k, v, do, True, scale, window=w)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = np.sum(oracle.forward_f64(*[xp if n == name else args[n] for n in "qkv"], True, scale,
                                           window=w)[0] * do)
            lm = np.sum(oracle.forward_f64(*[xm if n == name else args[n] for n in "qkv"], True, scale,
                                           window=w)[0] * do)
            assert abs((lp - lm) / (2 * h) - g[idx]) < 2e-7, (name, idx)


def test_window_needs_causal_and_a_key_per_row():
    q, k, v = make_qkv(1, 1, 8, 6, 8, seed_base=8600)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, True, 0.3, window=2)        # Lq > Lk
    q, k, v = make_qkv(1, 1, 6, 8, 8, seed_base=8601)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, False, 0.3, window=2)       # not causal
