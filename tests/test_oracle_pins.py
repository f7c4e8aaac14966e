"""Pins for the fp64 CPU oracle (no GPU).

The oracle (oracle/fa2_oracle.c) is the parity reference for the CUDA path, so
it is itself pinned to things other than itself:

  * hand-worked examples with rational answers (tests/golden/worked_examples.txt)
  * brute force in plain Python loops on tiny inputs (written independently)
  * a library routine for the same definition (torch SDPA / logsumexp, fp64)
  * closed forms: uniform scores, one-hot dominant scores, causal row 0
  * invariants: rows of P sum to 1 and vanish off the mask, LSE bounds,
    convexity of O, key-permutation invariance, homogeneity in V
  * mutation checks: plausible mistakes (no scale, wrong mask direction,
    swapped K/V, base-2 LSE, a dropped key, ...) each fail at least one pin.

Definition followed: O = softmax(scale Q K^T [+ causal mask]) V and
LSE_i = ln sum_j exp(s_ij) (Olowookere, "FlashAttention-2 from scratch with a
custom Triton kernel", section "The core idea: making attention IO-aware";
"Chapter 08: Flash Attention -- blocked attention", sections 3 and 4).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv, randn_bf16

HERE = os.path.dirname(os.path.abspath(__file__))
TINY = [  # (B, H, Lq, Lk, D)
    (1, 1, 1, 1, 1),
    (1, 1, 3, 3, 2),
    (2, 1, 5, 7, 4),
    (1, 2, 8, 8, 8),
    (2, 2, 6, 4, 3),
    (1, 1, 7, 5, 8),
]


# --------------------------------------------------------------------------
# implementations under test: the oracle, plus deliberately wrong variants
# --------------------------------------------------------------------------
def oracle_impl(q, k, v, causal, scale):
    return oracle.attention(q, k, v, causal, scale, threads=2)


def _np_attention(q, k, v, causal, scale, *, mutate=None):
    """numpy reference used ONLY to build mutated variants for the mutation test."""
    qd = q.double().numpy()
    kd = k.double().numpy()
    vd = v.double().numpy()
    if mutate == "swap_kv":
        kd, vd = vd, kd
    if mutate == "wrong_head":
        kd = np.roll(kd, 1, axis=1)
    s = np.einsum("bhid,bhjd->bhij", qd, kd)
    if mutate != "no_scale":
        s = s * scale
    Lq, Lk = s.shape[-2:]
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    vis = np.ones((Lq, Lk), bool)
    if causal:
        if mutate == "mask_strict":
            vis = j < i
            vis[:, 0] |= True  # keep rows non-empty so the variant stays finite
        elif mutate == "mask_flipped":
            vis = j >= i
        else:
            vis = j <= i
    if mutate == "drop_last_key":
        vis = vis & (j < Lk - 1) if Lk > 1 else vis
    s = np.where(vis, s, -np.inf)
    m = s.max(-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(-1, keepdims=True)
    p = e / z
    if mutate == "no_normalise":
        p = e
    o = p @ vd
    lse = (m + np.log(z))[..., 0]
    if mutate == "lse_base2":
        lse = lse / math.log(2.0)
    if mutate == "lse_no_max":
        lse = np.log(z)[..., 0]
    return o, lse


# --------------------------------------------------------------------------
# independent brute force: plain Python loops over lists of floats
# --------------------------------------------------------------------------
def brute_force(q, k, v, causal, scale):
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    Q, K, V = q.double().tolist(), k.double().tolist(), v.double().tolist()
    o = np.zeros((B, H, Lq, D))
    lse = np.zeros((B, H, Lq))
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                keys = [j for j in range(Lk) if (not causal) or j <= i]
                s = {j: scale * math.fsum(Q[b][h][i][d] * K[b][h][j][d] for d in range(D))
                     for j in keys}
                mx = max(s.values())
                w = {j: math.exp(s[j] - mx) for j in keys}
                z = math.fsum(w.values())
                for d in range(D):
                    o[b, h, i, d] = math.fsum(w[j] / z * V[b][h][j][d] for j in keys)
                lse[b, h, i] = mx + math.log(z)
    return o, lse


# --------------------------------------------------------------------------
# pin checks: each takes an implementation and returns a list of failures
# --------------------------------------------------------------------------
def _parse_golden():
    text = open(os.path.join(HERE, "golden", "worked_examples.txt")).read()
    blocks = []
    for raw in text.split("\n---"):
        fields = {}
        for line in raw.splitlines():
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            fields[key.strip()] = val.strip()
        if fields:
            blocks.append(fields)
    return blocks


def _rows(spec):
    return [[eval(x, {"math": math}) for x in r.split(",")] for r in spec.split(";")]


def check_golden(impl):
    bad = []
    for ex in _parse_golden():
        q = torch.tensor([[_rows(ex["q"])]], dtype=torch.float64).to(torch.bfloat16)
        k = torch.tensor([[_rows(ex["k"])]], dtype=torch.float64).to(torch.bfloat16)
        v = torch.tensor([[_rows(ex["v"])]], dtype=torch.float64).to(torch.bfloat16)
        # the fixture promises exact bf16 inputs
        assert torch.equal(q.double(), torch.tensor([[_rows(ex["q"])]], dtype=torch.float64))
        o_exp = np.array(_rows(ex["o"]))
        lse_exp = np.array([eval(x, {"math": math}) for x in ex["lse"].split(",")])
        o, lse = impl(q, k, v, bool(int(ex["causal"])), eval(ex["scale"], {"math": math}))
        o, lse = np.asarray(o)[0, 0], np.asarray(lse)[0, 0]
        if not (np.allclose(o, o_exp, rtol=0, atol=1e-12)
                and np.allclose(lse, lse_exp, rtol=0, atol=1e-12)):
            bad.append(ex["name"])
    return bad


def check_brute_force(impl):
    bad = []
    for n, (B, H, Lq, Lk, D) in enumerate(TINY):
        q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=77 + 10 * n)
        for causal in (False, True):
            scale = 1.0 / math.sqrt(D)
            o, lse = impl(q, k, v, causal, scale)
            o_ref, lse_ref = brute_force(q, k, v, causal, scale)
            if not (np.allclose(o, o_ref, rtol=0, atol=1e-12)
                    and np.allclose(lse, lse_ref, rtol=0, atol=1e-12)):
                bad.append((B, H, Lq, Lk, D, causal))
    return bad


def check_library(impl):
    """torch SDPA (fp64, CPU) for O and torch.logsumexp for LSE."""
    bad = []
    for n, (B, H, Lq, Lk, D) in enumerate(TINY + [(2, 3, 33, 47, 16)]):
        q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=500 + 10 * n)
        for causal in (False, True):
            scale = 0.37
            o, lse = impl(q, k, v, causal, scale)
            qd, kd, vd = q.double(), k.double(), v.double()
            o_ref = torch.nn.functional.scaled_dot_product_attention(
                qd, kd, vd, is_causal=causal, scale=scale).numpy()
            s = scale * qd @ kd.transpose(-1, -2)
            if causal:
                keep = torch.ones(Lq, Lk, dtype=torch.bool).tril()
                s = s.masked_fill(~keep, float("-inf"))
            lse_ref = torch.logsumexp(s, dim=-1).numpy()
            if not (np.allclose(o, o_ref, rtol=0, atol=1e-12)
                    and np.allclose(lse, lse_ref, rtol=0, atol=1e-12)):
                bad.append((B, H, Lq, Lk, D, causal))
    return bad


def check_uniform(impl):
    """Q = 0: every visible score is 0, so O_i = mean of visible V rows, LSE_i = ln|A_i|."""
    bad = []
    B, H, L, D = 1, 2, 9, 4
    _, k, v = make_qkv(B, H, L, L, D, seed_base=9)
    q = torch.zeros(B, H, L, D, dtype=torch.bfloat16)
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, 0.5)
        vd = v.double().numpy()
        for i in range(L):
            n = i + 1 if causal else L
            if not (np.allclose(o[:, :, i], vd[:, :, :n].mean(axis=2), rtol=0, atol=1e-12)
                    and np.allclose(lse[:, :, i], math.log(n), rtol=0, atol=1e-12)):
                bad.append((causal, i))
    return bad


def check_one_hot(impl):
    """Q_i = 64 e_pi(i), K_j = 64 e_j: score gap 4096*scale, O_i = V[pi(i)], LSE_i = 4096*scale."""
    bad = []
    D = 8
    L = 8
    scale = 1.0 / math.sqrt(D)
    rng = np.random.default_rng(3)
    for causal in (False, True):
        # causal needs pi(i) <= i; use the identity there, a permutation otherwise
        pi = np.arange(L) if causal else rng.permutation(L)
        q = torch.zeros(1, 1, L, D)
        k = torch.zeros(1, 1, L, D)
        for i in range(L):
            q[0, 0, i, pi[i]] = 64.0
            k[0, 0, i, i] = 64.0
        q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
        v = randn_bf16((1, 1, L, D), 11)
        o, lse = impl(q, k, v, causal, scale)
        vd = v.double().numpy()[0, 0]
        if not (np.allclose(o[0, 0], vd[pi], rtol=0, atol=1e-12)
                and np.allclose(lse[0, 0], 4096.0 * scale, rtol=0, atol=1e-9)):
            bad.append(causal)
    return bad


def check_causal_row0(impl):
    """Causal row 0 sees key 0 only: O_0 = V_0 exactly, LSE_0 = scale * q_0 . k_0."""
    q, k, v = make_qkv(2, 2, 6, 6, 5, seed_base=21)
    scale = 0.8
    o, lse = impl(q, k, v, True, scale)
    bad = []
    for b in range(2):
        for h in range(2):
            qr = q[b, h, 0].double().tolist()
            kr = k[b, h, 0].double().tolist()
            exp_lse = scale * math.fsum(a * c for a, c in zip(qr, kr))
            if not (np.array_equal(o[b, h, 0], v[b, h, 0].double().numpy())
                    and abs(lse[b, h, 0] - exp_lse) <= 1e-13):
                bad.append((b, h))
    return bad


def check_bounds_and_convexity(impl):
    """max_j s_ij <= LSE_i <= max_j s_ij + ln|A_i| and min_j v_jd <= O_id <= max_j v_jd."""
    bad = []
    q, k, v = make_qkv(1, 3, 12, 10, 6, seed_base=31)
    scale = 1.0 / math.sqrt(6)
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, scale)
        s = scale * (q.double() @ k.double().transpose(-1, -2)).numpy()
        vd = v.double().numpy()
        for h in range(3):
            for i in range(12):
                n = min(i + 1, 10) if causal else 10
                mx = s[0, h, i, :n].max()
                if not (mx - 1e-12 <= lse[0, h, i] <= mx + math.log(n) + 1e-12):
                    bad.append(("lse", causal, h, i))
                lo, hi = vd[0, h, :n].min(0), vd[0, h, :n].max(0)
                if not (np.all(o[0, h, i] >= lo - 1e-12) and np.all(o[0, h, i] <= hi + 1e-12)):
                    bad.append(("convex", causal, h, i))
    return bad


def check_permutation(impl):
    """Non-causal: permuting K and V rows together leaves O and LSE unchanged."""
    q, k, v = make_qkv(2, 2, 7, 11, 4, seed_base=41)
    perm = torch.randperm(11, generator=torch.Generator().manual_seed(5))
    o1, l1 = impl(q, k, v, False, 0.6)
    o2, l2 = impl(q, k[:, :, perm], v[:, :, perm], False, 0.6)
    ok = np.allclose(o1, o2, rtol=0, atol=1e-13) and np.allclose(l1, l2, rtol=0, atol=1e-13)
    return [] if ok else ["permutation"]


def check_homogeneity(impl):
    """V -> 2V gives O -> 2O exactly (doubling is exact in bf16 and fp64) and LSE unchanged."""
    q, k, v = make_qkv(1, 2, 5, 6, 3, seed_base=51)
    bad = []
    for causal in (False, True):
        o1, l1 = impl(q, k, v, causal, 0.9)
        o2, l2 = impl(q, k, v * 2, causal, 0.9)
        if not (np.array_equal(2 * o1, o2) and np.array_equal(l1, l2)):
            bad.append(causal)
    return bad


PIN_CHECKS = [check_golden, check_brute_force, check_library, check_uniform,
              check_one_hot, check_causal_row0, check_bounds_and_convexity,
              check_permutation, check_homogeneity]


# --------------------------------------------------------------------------
# the pins, applied to the oracle
# --------------------------------------------------------------------------
@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    assert check(oracle_impl) == []


def test_decode_bf16_all_patterns():
    """The oracle's bf16 -> fp64 widening matches torch's for all 65536 bit patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref, equal_nan=True)


def test_p_rows_are_distributions():
    """Materialised P rows: sum to 1, lie in [0, 1], vanish exactly off the causal mask."""
    B, H, Lq, Lk, D = 2, 2, 9, 13, 8
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=61)
    for causal in (False, True):
        rows = np.arange(B * H * Lq, dtype=np.int64)
        _, _, p = oracle.attention_rows(q, k, v, causal, 0.35, rows, return_p=True)
        assert np.all(p >= 0) and np.all(p <= 1)
        assert np.allclose(p.sum(1), 1.0, rtol=0, atol=1e-12)
        if causal:
            i = rows % Lq
            j = np.arange(Lk)[None, :]
            assert np.all(p[j > i[:, None]] == 0.0)
            assert np.all(p[j <= i[:, None]] > 0.0)


def test_row_subset_matches_full():
    """Rows computed on their own equal the same rows of a full evaluation, bit for bit."""
    q, k, v = make_qkv(2, 3, 17, 19, 8, seed_base=71)
    o_full, l_full = oracle.attention(q, k, v, True, 0.4)
    rows = np.array([0, 5, 16, 17, 40, 101], dtype=np.int64)
    o, l = oracle.attention_rows(q, k, v, True, 0.4, rows)
    assert np.array_equal(o, o_full.reshape(-1, 8)[rows])
    assert np.array_equal(l, l_full.reshape(-1)[rows])


def test_rejects_bad_rows():
    q, k, v = make_qkv(1, 1, 4, 4, 2, seed_base=1)
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, k, v, False, 1.0, np.array([4], dtype=np.int64))


MUTATIONS = ["no_scale", "mask_strict", "mask_flipped", "swap_kv", "wrong_head",
             "drop_last_key", "no_normalise", "lse_base2", "lse_no_max"]


def test_numpy_variant_unmutated_passes():
    """Sanity for the mutation test: the unmutated numpy variant passes every pin."""
    impl = lambda q, k, v, c, s: _np_attention(q, k, v, c, s)  # noqa: E731
    for check in PIN_CHECKS:
        assert check(impl) == [], check.__name__


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_catch_planted_mistake(mutation):
    """Each plausible mistake fails at least one pin, so the pins constrain the oracle."""
    impl = lambda q, k, v, c, s: _np_attention(q, k, v, c, s, mutate=mutation)  # noqa: E731
    caught = []
    for check in PIN_CHECKS:
        with np.errstate(all="ignore"):
            if check(impl):
                caught.append(check.__name__)
    assert caught, f"no pin catches mutation {mutation}"
