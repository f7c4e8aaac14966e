"""A seeded sweep of random problem shapes, forward and backward, against the oracle
("Chapter 08: Flash Attention -- blocked attention", sections 3-6): batch, heads, query
and key lengths (1 to 1200 forward, 900 backward: ragged against every tile size), head dimension, causal or
not, the query scaled by 1 or 2 (peakier rows, more rescales of O), and for non-causal
passes the workspace path with the key-tile ranges cut at every SM (FA2_SPLIT=always).
Every element is compared: O and LSE with the forward's bar, dQ, dK and dV with the
backward's (relative rms and largest error per tensor)."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv
from parity import compare
from test_bwd_gpu import compare_grads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _cases(n, seed, max_len):
    rng = np.random.RandomState(seed)
    out = []
    for i in range(n):
        B, H = int(rng.randint(1, 4)), int(rng.randint(1, 5))
        Lq, Lk = int(rng.randint(1, max_len + 1)), int(rng.randint(1, max_len + 1))
        D = int(rng.choice([64, 128, 256]))
        causal = bool(rng.randint(0, 2))
        qmul = float(rng.choice([1.0, 2.0]))
        split = (not causal) and bool(rng.randint(0, 2))
        out.append((i, B, H, Lq, Lk, D, causal, qmul, split))
    return out


FWD = _cases(64, 2027, 1200)
BWD = [c[:7] for c in _cases(24, 2028, 900)]


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal,qmul,split", FWD)
def test_forward_random_shape(i, B, H, Lq, Lk, D, causal, qmul, split, monkeypatch):
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_get_device_error, fa2_workspace
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=12000 + 10 * i)
    if qmul != 1.0:
        q = (q.float() * qmul).to(torch.bfloat16)   # exact: a power of two
    scale = D ** -0.5
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if split:
        monkeypatch.setenv("FA2_SPLIT", "always")
        ws = fa2_workspace(qd, kd, causal)
    fa2_fwd(qd, kd, vd, o, lse, causal, scale, workspace=ws)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref)


@pytest.mark.parametrize("i,B,H,Lq,Lk,D,causal", BWD)
def test_backward_random_shape(i, B, H, Lq, Lk, D, causal):
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_fwd, fa2_get_device_error
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=13000 + 10 * i)
    do = make_qkv(B, H, Lq, Lq, D, seed_base=13500 + 10 * i)[0]
    scale = D ** -0.5
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device=DEV)
    fa2_fwd(qd, kd, vd, o, lse, causal, scale)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    fa2_bwd(qd, kd, vd, o, lse, dod, *grads, causal, scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    compare_grads((q, k, v, do, scale), [g.cpu() for g in grads], causal)
