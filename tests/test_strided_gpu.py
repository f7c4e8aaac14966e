"""GPU parity of the strided entry point fa2_fwd_ex ("FlashAttention-2 from scratch
with a custom Triton kernel", host wrapper and kernel launch: the kernel is given
every tensor's strides).

Only the addressing differs from the contiguous path: TMA descriptors built from
the views' strides, and O rows stored at their strided addresses.  So every case is
checked bit for bit against fa2_fwd on contiguous copies of the same values, and
a few also against the fp64 oracle.
"""
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv
from parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _contiguous_run(q, k, v, causal, scale, window=None):
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_fwd_window
    B, H, Lq, D = q.shape
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=DEV)
    qc, kc, vc = (t.contiguous() for t in (q, k, v))
    if window is None:
        fa2_fwd(qc, kc, vc, o, lse, causal, scale)
    else:
        fa2_fwd_window(qc, kc, vc, o, lse, window, scale)
    return o, lse


def _strided_run(q, k, v, o_view, causal, scale, window=None, workspace=None):
    from io_aware_exact_fa2_gb300 import fa2_fwd_ex, fa2_get_device_error
    B, H, Lq, D = q.shape
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=DEV)
    o_view.fill_(float("nan"))
    fa2_fwd_ex(q, k, v, o_view, lse, causal, scale, window=window, workspace=workspace)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error status {st} code {code:#x}"
    return o_view, lse


def _blhd(t):
    """The same values stored as [B, L, H, D] and viewed as [B, H, L, D]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_blhd_views_match_contiguous(D, causal):
    B, H, Lq, Lk = 2, 3, 300, 457 if not causal else 300
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, Lq, Lk, D, seed_base=9100 + D))
    scale = D ** -0.5
    o_ref, lse_ref = _contiguous_run(q, k, v, causal, scale)
    o_store = torch.empty(B, Lq, H, D, dtype=torch.bfloat16, device=DEV)   # O also as [B, L, H, D]
    o, lse = _strided_run(_blhd(q), _blhd(k), _blhd(v), o_store.transpose(1, 2), causal, scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_packed_qkv_slices_and_padded_o_against_oracle(causal):
    """q, k, v as slices of one packed [B, L, 3, H, D] tensor; O written into every
    other row of a wider buffer; checked against the oracle and the contiguous path."""
    B, H, L, D = 1, 4, 389, 128
    qh, kh, vh = make_qkv(B, H, L, L, D, seed_base=9200)
    packed = torch.stack([t.transpose(1, 2) for t in (qh, kh, vh)], dim=2).contiguous().to(DEV)
    q, k, v = (packed[:, :, i].transpose(1, 2) for i in range(3))
    assert q.stride(2) == 3 * H * D
    scale = D ** -0.5
    wide = torch.empty(B, H, 2 * L, D, dtype=torch.bfloat16, device=DEV)
    o_view = wide[:, :, ::2]
    o, lse = _strided_run(q, k, v, o_view, causal, scale)
    o_c, lse_c = _contiguous_run(q, k, v, causal, scale)
    assert torch.equal(o, o_c) and torch.equal(lse, lse_c)
    o_ref, lse_ref = oracle.attention(qh, kh, vh, causal, scale)
    compare(o.contiguous().cpu(), lse.cpu(), o_ref, lse_ref)


def test_split_schedule_with_strided_views():
    """Non-causal with a workspace (cost-balanced ranges, cut units merged) on BLHD views."""
    from io_aware_exact_fa2_gb300 import fa2_workspace_size
    B, H, L, D = 2, 16, 1536, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed_base=9300))
    n = fa2_workspace_size(B, H, L, L, D, False)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=DEV)
    o_ref, lse_ref = _contiguous_run(q, k, v, False, D ** -0.5)
    o_store = torch.empty(B, L, H, D, dtype=torch.bfloat16, device=DEV)
    o, lse = _strided_run(_blhd(q), _blhd(k), _blhd(v), o_store.transpose(1, 2), False, D ** -0.5, workspace=ws)
    # the split schedule sums parts in another order than whole units: compare to the oracle
    # on sampled heads, and to the contiguous path within the parity tolerance
    assert float((o.float() - o_ref.float()).abs().max()) <= 1e-2
    assert float((lse - lse_ref).abs().max()) <= 1e-3
    qh, kh, vh = (t.cpu() for t in (q, k, v))
    for bh in (0, 17, 31):
        b, h = divmod(bh, H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_r, l_r = oracle.attention(qh[sl], kh[sl], vh[sl], False, D ** -0.5)
        compare(o[sl].contiguous().cpu(), lse[sl].cpu(), o_r, l_r)


def test_window_with_strided_views():
    B, H, L, D, w = 1, 2, 700, 64, 100
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed_base=9400))
    o_ref, lse_ref = _contiguous_run(q, k, v, True, D ** -0.5, window=w)
    o_store = torch.empty(B, L, H, D, dtype=torch.bfloat16, device=DEV)
    o, lse = _strided_run(_blhd(q), _blhd(k), _blhd(v), o_store.transpose(1, 2), True, D ** -0.5, window=w)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_rejects_unaligned_strides():
    from io_aware_exact_fa2_gb300 import Fa2Error, fa2_fwd_ex
    B, H, L, D = 1, 2, 64, 64
    base = torch.zeros(B, H, L, D + 4, dtype=torch.bfloat16, device=DEV)
    q = base[..., :D]                     # row stride 68 elements: not a multiple of 16 bytes
    o = torch.empty(B, H, L, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, L, dtype=torch.float32, device=DEV)
    with pytest.raises(Fa2Error):
        fa2_fwd_ex(q, q, q, o, lse, False)


# ---------------------------------------------------------------- backward (fa2_bwd_ex)
def _contiguous_bwd(q, k, v, do, causal, scale, window=None):
    """Forward and backward on contiguous copies: (o, lse, dq, dk, dv)."""
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_bwd_window
    qc, kc, vc, dc = (t.contiguous() for t in (q, k, v, do))
    o, lse = _contiguous_run(qc, kc, vc, causal, scale, window)
    grads = [torch.full_like(t, float("nan")) for t in (qc, kc, vc)]
    if window is None:
        fa2_bwd(qc, kc, vc, o, lse, dc, *grads, causal, scale)
    else:
        fa2_bwd_window(qc, kc, vc, o, lse, dc, *grads, window, scale)
    return (o, lse, *grads)


def _strided_bwd(q, k, v, do, o, lse, grads, causal, scale, window=None):
    from io_aware_exact_fa2_gb300 import fa2_bwd_ex, fa2_get_device_error
    for g in grads:
        g.fill_(float("nan"))
    fa2_bwd_ex(q, k, v, o, lse, do, *grads, causal, scale, window=window)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {st} code {code:#x}"
    return grads


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_bwd_blhd_views_match_contiguous(D, causal):
    """Every tensor of the backward stored as [B, L, H, D] and viewed as [B, H, L, D]:
    bit-identical to fa2_bwd on contiguous copies."""
    B, H, Lq, Lk = 2, 3, 300, 457 if not causal else 300
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, Lq, Lk, D, seed_base=9600 + D))
    do = make_qkv(B, H, Lq, Lq, D, seed_base=9650 + D)[0].to(DEV)
    scale = D ** -0.5
    o, lse, *ref = _contiguous_bwd(q, k, v, do, causal, scale)
    grads = [torch.empty(B, L, H, D, dtype=torch.bfloat16, device=DEV).transpose(1, 2) for L in (Lq, Lk, Lk)]
    got = _strided_bwd(_blhd(q), _blhd(k), _blhd(v), _blhd(do), _blhd(o), lse, grads, causal, scale)
    for g, r in zip(got, ref):
        assert torch.equal(g, r)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_bwd_packed_qkv_and_packed_gradients(causal):
    """q, k, v as slices of one packed [B, L, 3, H, D] tensor and dq, dk, dv written into the
    slices of one packed gradient tensor of the same layout; bit-identical to the contiguous
    backward, and checked against the oracle's gradients."""
    B, H, L, D = 1, 4, 389, 128
    qh, kh, vh = make_qkv(B, H, L, L, D, seed_base=9700)
    doh = make_qkv(B, H, L, L, D, seed_base=9750)[0]
    packed = torch.stack([t.transpose(1, 2) for t in (qh, kh, vh)], dim=2).contiguous().to(DEV)
    q, k, v = (packed[:, :, i].transpose(1, 2) for i in range(3))
    do = doh.to(DEV)
    scale = D ** -0.5
    o, lse, *ref = _contiguous_bwd(q, k, v, do, causal, scale)
    gpacked = torch.empty(B, L, 3, H, D, dtype=torch.bfloat16, device=DEV)
    grads = [gpacked[:, :, i].transpose(1, 2) for i in range(3)]
    got = _strided_bwd(q, k, v, do, o, lse, grads, causal, scale)
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
    from test_bwd_gpu import compare_grads
    compare_grads((qh, kh, vh, doh, scale), [g.contiguous().cpu() for g in got], causal)


def test_bwd_window_with_strided_views():
    B, H, L, D, w = 1, 2, 700, 64, 100
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed_base=9800))
    do = make_qkv(B, H, L, L, D, seed_base=9850)[0].to(DEV)
    o, lse, *ref = _contiguous_bwd(q, k, v, do, True, D ** -0.5, window=w)
    grads = [torch.empty(B, L, H, D, dtype=torch.bfloat16, device=DEV).transpose(1, 2) for _ in range(3)]
    got = _strided_bwd(_blhd(q), _blhd(k), _blhd(v), _blhd(do), _blhd(o), lse, grads, True, D ** -0.5, window=w)
    for g, r in zip(got, ref):
        assert torch.equal(g, r)


def test_bwd_no_queries_zeroes_strided_key_gradients():
    """Lq = 0: dk and dv are zeroed row by row in their strided views, and nothing else moves
    (the query-side buffers are never read; dummies stand in for the empty tensors)."""
    import ctypes
    from io_aware_exact_fa2_gb300 import _binding
    B, H, Lk, D = 2, 3, 50, 64
    k = torch.randn(B, H, Lk, D, device=DEV).to(torch.bfloat16)
    dummy = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(4, dtype=torch.float32, device=DEV)
    wide = torch.full((B, Lk, H, 2 * D), 7.0, dtype=torch.bfloat16, device=DEV)
    dk = wide[..., :D].transpose(1, 2)           # rows 2*D elements apart; the other half must stay 7
    dv = torch.full((B, H, Lk, D), 7.0, dtype=torch.bfloat16, device=DEV)
    ll3 = ctypes.c_longlong * 3
    strides = [None] * 6 + [ll3(dk.stride(0), dk.stride(1), dk.stride(2)), None]
    p = dummy.data_ptr()
    st = _binding._lib.fa2_bwd_ex(p, k.data_ptr(), k.data_ptr(), p, lse.data_ptr(), p, p, dk.data_ptr(),
                                  dv.data_ptr(), B, H, 0, Lk, D, *strides, 0, -1, 0.125, None, 0, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0
    assert bool((wide[..., D:] == 7.0).all())
