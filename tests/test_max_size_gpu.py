"""GPU parity past 2^31 elements per tensor.

The shape is B=2, H=10000, L=1024, D=128: 2.62e9 elements (5.2 GB of bf16) per tensor.
Heads from b=1, h=6384 on start past element 2^31, and every head from b=0, h=8192 on
starts past byte 2^32. So the addressing of every buffer (TMA maps over (D, L, H, B),
O and LSE rows, the backward's statistics tiles and gradient rows) is exercised past
32-bit offsets. Sampled heads, first and last included, are checked against the fp64
oracle, the forward with the parity tolerance of the other forward tests (tests/parity.py)
and the backward with the tolerance of the backward tests.

The inputs are built without generating 8e9 random numbers on the host. A seeded CPU
base of 64 heads is drawn from the shared input generator, and head bh of the large
tensors is base head bh mod 64 rolled by bh // 64 rows along L. All 20000 heads
therefore differ, so reading a wrong head cannot go unnoticed. The GPU builds the
large tensors with a torch gather. The oracle gets the same construction done on the
CPU from the same base; it takes nothing from the GPU but the outputs under test.
"""
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import make_qkv
from parity import compare
from test_bwd_gpu import compare_grads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
B, H, L, D = 2, 10000, 1024, 128
NBASE = 64
assert B * H * L * D > 2 ** 31
HEADS = [(0, 0), (0, 8191), (0, 8192), (1, 6383), (1, 6384), (1, H - 1)]


def _base(seed):
    q, k, v = make_qkv(1, NBASE, L, L, D, seed_base=seed)
    do = make_qkv(1, NBASE, L, L, D, seed_base=seed + 500)[0]
    return [t[0] for t in (q, k, v, do)]          # [NBASE, L, D] each


def _head_cpu(base, bh):
    """Head bh of the large tensor, built on the CPU: base head bh % 64 rolled by bh // 64 rows."""
    return torch.roll(base[bh % NBASE], bh // NBASE, dims=0)[None, None]


def _large_gpu(base):
    """All B*H heads on the GPU: out[bh, l] = base[bh % 64, (l - bh // 64) mod L]."""
    bd = base.to(DEV)
    bh = torch.arange(B * H, device=DEV)
    rows = (torch.arange(L, device=DEV)[None, :] - (bh // NBASE)[:, None]) % L
    out = bd[(bh % NBASE)[:, None], rows]
    del bd, rows
    return out.view(B, H, L, D)


@pytest.fixture(scope="module")
def inputs():
    base = _base(9600)
    big = [_large_gpu(t) for t in base]
    # the GPU construction matches the CPU one on the sampled heads
    for b, h in HEADS:
        for t, bt in zip(big, base):
            assert torch.equal(t[b, h].cpu(), _head_cpu(bt, b * H + h)[0, 0])
    yield base, big
    del big
    torch.cuda.empty_cache()


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_forward_past_2_31_elements(inputs, causal):
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_get_device_error
    base, (q, k, v, _) = inputs
    scale = D ** -0.5
    o = torch.full((B, H, L, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, L), float("nan"), dtype=torch.float32, device=DEV)
    fa2_fwd(q, k, v, o, lse, causal, scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {st} code {code:#x}"
    for b, h in HEADS:
        bh = b * H + h
        o_ref, lse_ref = oracle.attention(*(_head_cpu(t, bh) for t in base[:3]), causal, scale)
        compare(o[b:b + 1, h:h + 1].cpu(), lse[b:b + 1, h:h + 1].cpu(), o_ref, lse_ref)
    del o, lse


def test_backward_past_2_31_elements(inputs):
    from io_aware_exact_fa2_gb300 import fa2_bwd, fa2_fwd, fa2_get_device_error
    base, (q, k, v, do) = inputs
    scale = D ** -0.5
    o = torch.empty((B, H, L, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=DEV)
    fa2_fwd(q, k, v, o, lse, False, scale)
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    fa2_bwd(q, k, v, o, lse, do, *grads, False, scale)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {st} code {code:#x}"
    del o, lse
    for b, h in HEADS[::2] + [HEADS[-1]]:
        bh = b * H + h
        head_in = [_head_cpu(t, bh) for t in base]
        got = [g[b:b + 1, h:h + 1].cpu() for g in grads]
        compare_grads((*head_in, scale), got, False)
