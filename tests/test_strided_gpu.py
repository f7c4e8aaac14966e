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
