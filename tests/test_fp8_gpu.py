"""FP8 forward (fa2_fwd_fp8) on the GPU against the oracle's exact attention of the
dequantised inputs ("Flash Attention: principles and implementation", section 4.3,
names FlashAttention-3's FP8 mode; the reading taken is e4m3 Q, K, V with one fp32
descale per (batch, head) each).

Tolerance, from the arithmetic.  The products Q K^T and P V accumulate exactly
representable e4m3 products in fp32, so the scores are as good as fp32.  What the
FP8 path adds is the rounding of the softmax weights to e4m3 for the P V product.
The kernel's weights are p_j = 2^(x_j - m) with m its running reference max (at or
below the row max M, by less than 2^8); a weight in e4m3's normal range (p >= 2^-6)
rounds by at most 2^-4 of itself, a smaller one by at most 2^-10 (half the 2^-9
subnormal spacing; the smallest round to zero).  O is divided by the sum of the
rounded weights p~, so exactly

    O_gpu - O = sum_j (p~_j - p_j)(v_j - O) / sum_j p~_j,   sum_j p~_j >= (1 - 2^-4) sum_j p_j.

With r_j = 2^(x_j - M) (so p_j >= r_j, and only keys with r_j < 2^-6 can be
subnormal) and w_j = r_j / sum r the exact weights, per element

    |dO_d| <= b_d = [2^-4 sum_j w_j |v_jd - O_d| + 2^-10 sum_{r_j < 2^-6} |v_jd - O_d| / sum_j r_j] / (1 - 2^-4),

and storing O in bf16 adds at most 2^-8 (|O_d| + b_d); 1e-4 covers the fp32
accumulation.  LSE comes from the unrounded fp32 sum and keeps the bf16 path's
1e-3.  b_d is computed per checked row from the exact scores (fp64, numpy, on the
dequantised inputs).  A CPU simulation of the kernel's rounding (reference max at
0, 3.3 and 7.9 below the row max) stays within 0.8 of this bound on these shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv_fp8
from parity import sample_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_fp8(q8, k8, v8, dq, dk, dv, causal, scale, workspace=False):
    from io_aware_exact_fa2_gb300 import fa2_fwd_fp8, fa2_get_device_error, fa2_workspace_size
    B, H, Lq, D = q8.shape
    Lk = k8.shape[2]
    args = [t.to(DEV) for t in (q8, k8, v8)] + [torch.from_numpy(d).to(DEV) for d in (dq, dk, dv)]
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if workspace:
        n = fa2_workspace_size(B, H, Lq, Lk, 128, causal)
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=DEV)
    fa2_fwd_fp8(*args, o, lse, causal, scale, workspace=ws)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    return o.cpu(), lse.cpu()


def o_bound(q, k, v, causal, scale, rows):
    """Per-element bound of the docstring for flat rows `rows`, from the exact weights."""
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    out = np.empty((len(rows), D))
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), Lq)
        b, h = divmod(bh, H)
        kk, vv = k[b, h], v[b, h]
        last = min(i, Lk - 1) if causal else Lk - 1
        s = scale * (kk[:last + 1] @ q[b, h, i])
        rw = np.exp(s - s.max())
        w = rw / rw.sum()
        o = w @ vv[:last + 1]
        dev = np.abs(vv[:last + 1] - o)
        bd = (2.0 ** -4 * (w @ dev) + 2.0 ** -10 * ((rw < 2.0 ** -6) @ dev) / rw.sum()) / (1 - 2.0 ** -4)
        out[n] = bd + 2.0 ** -8 * (np.abs(o) + bd) + 1e-4
    return out


def check(q8, k8, v8, dq, dk, dv, causal, o, lse, rows):
    scale = q8.shape[-1] ** -0.5
    o_ref, lse_ref = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, causal, scale, rows)
    idx = torch.from_numpy(rows)
    og = o.double().reshape(-1, o.shape[-1])[idx].numpy()
    lg = lse.double().reshape(-1)[idx].numpy()
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    assert np.max(np.abs(lg - lse_ref)) <= 1e-3, np.max(np.abs(lg - lse_ref))
    q, k, v = (oracle.dequant_e4m3(t, d) for t, d in ((q8, dq), (k8, dk), (v8, dv)))
    bound = o_bound(q, k, v, causal, scale, rows)
    err = np.abs(og - o_ref)
    assert np.all(err <= bound), (float(err.max()), float((err - bound).max()))
    return float(err.max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 3, 300, 457), (1, 2, 129, 130), (2, 2, 640, 640), (1, 1, 1, 77)])
def test_fp8_every_element(shape, causal):
    B, H, Lq, Lk = shape
    q8, k8, v8, dq, dk, dv = make_qkv_fp8(B, H, Lq, Lk, 128, seed_base=8000 + Lq)
    o, lse = run_fp8(q8, k8, v8, dq, dk, dv, causal, 128 ** -0.5)
    check(q8, k8, v8, dq, dk, dv, causal, o, lse, np.arange(B * H * Lq, dtype=np.int64))


def test_fp8_split_schedule_matches_whole_tiles(monkeypatch):
    """Non-causal with the key-tile ranges cut at every SM (workspace, FA2_SPLIT=always):
    the parts merge into the same attention (checked against the oracle)."""
    monkeypatch.setenv("FA2_SPLIT", "always")
    q8, k8, v8, dq, dk, dv = make_qkv_fp8(1, 4, 1000, 4096, 128, seed_base=8100)
    o, lse = run_fp8(q8, k8, v8, dq, dk, dv, False, 128 ** -0.5, workspace=True)
    check(q8, k8, v8, dq, dk, dv, False, o, lse, np.arange(4 * 1000, dtype=np.int64))


@pytest.mark.parametrize("name,causal", [("c3", False), ("c3", True), ("c4", True)])
def test_fp8_at_the_bf16_workload_shapes(name, causal):
    """B2 H16 L4096 and B1 H32 L16384 (D = 128): tile edges of the first and last head plus
    random rows against the derived bound; every row finite; causal row 0 equals V_0."""
    B, H, L = (2, 16, 4096) if name == "c3" else (1, 32, 16384)
    q8, k8, v8, dq, dk, dv = make_qkv_fp8(B, H, L, L, 128, seed_base=8200 + L)
    o, lse = run_fp8(q8, k8, v8, dq, dk, dv, causal, 128 ** -0.5, workspace=not causal)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    if causal:   # row 0 sees key 0 alone: O_0 = dv * V8_0 up to the bf16 rounding of O
        v0 = v8[:, :, 0].double() * torch.from_numpy(dv).double()[:, :, None]
        assert torch.allclose(o[:, :, 0].double(), v0, rtol=2.0 ** -8, atol=0)
    rows = sample_rows(B, H, L, n_random=384, seed=8300 + L + int(causal))
    err = check(q8, k8, v8, dq, dk, dv, causal, o, lse, rows)
    print(f"fp8 {name} causal={causal}: max|dO| {err:.3e} over {len(rows)} rows")


def test_fp8_rejects_other_head_dims_and_missing_descales():
    from io_aware_exact_fa2_gb300 import Fa2Error, fa2_fwd_fp8
    q8, k8, v8, dq, dk, dv = make_qkv_fp8(1, 1, 16, 16, 64, seed_base=1)
    args = [t.to(DEV) for t in (q8, k8, v8)] + [torch.from_numpy(d).to(DEV) for d in (dq, dk, dv)]
    o = torch.empty(1, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 1, 16, dtype=torch.float32, device=DEV)
    with pytest.raises(Fa2Error) as e:
        fa2_fwd_fp8(*args, o, lse, False)
    assert e.value.status == 2   # FA2_ERR_UNSUPPORTED
