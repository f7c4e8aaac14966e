"""Pins for the oracle's FP8 path (no GPU).

"Flash Attention: principles and implementation" (tbr8.org), section 4.3, names
FlashAttention-3's FP8 mode without fixing a format.  The reading taken: Q, K and V
are stored as e4m3 with one fp32 descale per (batch, head) each, the real input
being stored value x descale; the reference is exact attention of those real
inputs.  The oracle's FP8 path therefore has two parts of its own, each pinned to
something other than itself:

  * the e4m3 widening: against torch's float8_e4m3fn conversion for all 256 codes,
    and against values worked out by hand from the format definition;
  * the dequantisation by per-(batch, head) descales: every e4m3 value is also a
    bf16 value, so with unit descales the FP8 path must reproduce the (already
    pinned) bf16 oracle bit for bit; powers-of-two descales must act exactly as
    the definition says (on V: O scales; on Q or K: the same as scaling the
    softmax scale); a descale of one head touches that head only; and the
    uniform-score closed form (Q = 0: O is the mean of the visible V rows).
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv_fp8


def test_decode_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours, ref, equal_nan=True)


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x80, -0.0), (0x38, 1.0), (0xB8, -1.0), (0x40, 2.0), (0x3C, 1.5),
    (0x7E, 448.0),             # largest finite: exponent 15, mantissa 6: 1.75 * 2^8
    (0x08, 2.0 ** -6),         # smallest normal
    (0x01, 2.0 ** -9),         # smallest subnormal: 1/8 * 2^-6
    (0x07, 7 * 2.0 ** -9),     # largest subnormal
])
def test_decode_e4m3_worked_values(code, value):
    got = oracle.decode_e4m3(np.array([code], dtype=np.uint8))[0]
    assert got == value and np.signbit(got) == np.signbit(value)


def test_decode_e4m3_nan_codes():
    got = oracle.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(got).all()


def _fp8_case(B, H, Lq, Lk, D, seed):
    q8, k8, v8, dq, dk, dv = make_qkv_fp8(B, H, Lq, Lk, D, seed_base=seed)
    return q8, k8, v8, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_unit_descales_reproduce_the_bf16_oracle(causal):
    """e4m3 values are bf16 values: with descales 1 the FP8 path equals the bf16 path exactly."""
    q8, k8, v8, _, _, _ = _fp8_case(2, 3, 9, 13, 16, 301)
    ones = np.ones((2, 3), dtype=np.float32)
    o8, l8 = oracle.attention_fp8(q8, k8, v8, ones, ones, ones, causal, 0.3)
    qb, kb, vb = (t.float().to(torch.bfloat16) for t in (q8, k8, v8))
    assert torch.equal(qb.float(), q8.float())   # the cast to bf16 was exact
    ob, lb = oracle.attention(qb, kb, vb, causal, 0.3)
    assert np.array_equal(o8, ob.reshape(-1, 16)) and np.array_equal(l8, lb.reshape(-1))


def test_descale_laws():
    q8, k8, v8, dq, dk, dv = _fp8_case(2, 2, 7, 11, 8, 311)
    o, l = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, False, 0.25)
    # V's descale doubled: O doubles exactly, LSE unchanged
    o2, l2 = oracle.attention_fp8(q8, k8, v8, dq, dk, 2 * dv, False, 0.25)
    assert np.array_equal(o2, 2 * o) and np.array_equal(l2, l)
    # Q's descale doubled and the scale halved: the same scores, bit for bit
    o3, l3 = oracle.attention_fp8(q8, k8, v8, 2 * dq, dk, dv, False, 0.125)
    assert np.array_equal(o3, o) and np.array_equal(l3, l)
    # K's descale quadrupled equals the scale quadrupled
    o4, l4 = oracle.attention_fp8(q8, k8, v8, dq, 4 * dk, dv, False, 0.25)
    o5, l5 = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, False, 1.0)
    assert np.array_equal(o4, o5) and np.array_equal(l4, l5)


def test_descale_is_per_batch_and_head():
    """Changing one (batch, head)'s descales changes that head's rows only."""
    B, H, Lq, Lk, D = 2, 3, 5, 6, 8
    q8, k8, v8, dq, dk, dv = _fp8_case(B, H, Lq, Lk, D, 321)
    o, l = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, True, 0.5)
    dq2, dv2 = dq.copy(), dv.copy()
    dq2[1, 2] *= 3.0
    dv2[1, 2] *= 0.5
    o2, l2 = oracle.attention_fp8(q8, k8, v8, dq2, dk, dv2, True, 0.5)
    heads = np.repeat(np.arange(B * H), Lq)
    changed = heads == 1 * H + 2
    assert np.array_equal(o2[~changed], o[~changed]) and np.array_equal(l2[~changed], l[~changed])
    assert not np.allclose(o2[changed], o[changed])


def test_uniform_scores_give_the_mean_of_v():
    """Q = 0 (stored zeros): every visible key has weight 1/|A_i|, so O is the mean of the
    dequantised V rows and LSE = ln |A_i|."""
    B, H, Lq, Lk, D = 1, 2, 6, 6, 8
    _, k8, v8, _, dk, dv = _fp8_case(B, H, Lq, Lk, D, 331)
    q8 = torch.zeros(B, H, Lq, D).to(torch.float8_e4m3fn)
    dq = np.ones((B, H), dtype=np.float32)
    o, l = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, True, 0.7)
    vr = v8.double().numpy() * dv[:, :, None, None].astype(np.float64)
    for bh in range(B * H):
        b, h = divmod(bh, H)
        for i in range(Lq):
            np.testing.assert_allclose(o[bh * Lq + i], vr[b, h, :i + 1].mean(0), rtol=0, atol=1e-14)
            assert abs(l[bh * Lq + i] - np.log(i + 1)) < 1e-14
