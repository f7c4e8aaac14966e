"""CUDA path vs the fp64 oracle, element by element, at sizes the oracle finishes
in seconds: several tiles, ragged tails, every head dimension, both mask modes,
Lq != Lk, single rows/keys, plus determinism, stream and bounds checks."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import WORKLOADS, make_qkv, workload_inputs
from parity import compare, run_cuda, sample_rows, scale_of

pytestmark = pytest.mark.gpu


def check(B, H, Lq, Lk, D, causal, seed, peaky_every=0):
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed, peaky_every=peaky_every)
    scale = scale_of(D)
    o, lse = run_cuda(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    return compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_c1_full(causal):
    """B1 H2 L128 D64: the small workload, every output element."""
    w = WORKLOADS["c1"]
    q, k, v = workload_inputs(w)
    o, lse = run_cuda(q, k, v, causal, w.scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, w.scale)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_ragged_multi_tile(D, causal):
    """Lq, Lk not multiples of any tile: partial Q groups, partial key tiles."""
    check(1, 2, 300, 457, D, causal, seed=100 + D)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_causal_square_several_tiles(D):
    check(2, 3, 640, 640, D, True, seed=200 + D)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Lq,Lk", [(200, 100), (100, 300), (513, 129)])
def test_causal_lq_ne_lk(D, Lq, Lk):
    """Top-left causal rule j <= i when Lq != Lk."""
    check(1, 2, Lq, Lk, D, True, seed=300 + Lq + Lk + D)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Lq,Lk", [(1, 1), (1, 1000), (129, 1), (257, 64), (2, 3)])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_degenerate_sizes(D, Lq, Lk, causal):
    check(1, 1, Lq, Lk, D, causal, seed=400 + Lq + Lk)


def test_peaky_rows_d256():
    """The peaky-key recipe (every 64th key x8) at a reduced size, non-causal."""
    check(1, 2, 400, 700, 256, False, seed=5000, peaky_every=64)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_many_heads_small_seq(D):
    check(3, 5, 130, 190, D, False, seed=600 + D)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_many_units_per_cta(D, causal):
    """More work units than SMs, with ragged Lq/Lk, so each persistent CTA walks several
    units (phases carried across units, Q/K/V prefetched for the next unit)."""
    check(8, 20, 300, 457, D, causal, seed=650 + D)


def run_ws(q, k, v, causal, scale, ws=None):
    """fa2_fwd_ws on seeded CPU inputs (workspace from fa2_workspace unless given)."""
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_get_device_error, fa2_workspace
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, H, Lq, D = q.shape
    if ws is None:
        ws = fa2_workspace(qd, kd, causal)
    o = torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=dev)
    fa2_fwd(qd, kd, vd, o, lse, causal, scale, workspace=ws)
    st, code = fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    return o.cpu(), lse.cpu(), ws


@pytest.fixture
def split_always(monkeypatch):
    """Force the cut-range schedule whenever a workspace is given (small shapes
    would otherwise be estimated not to gain from it)."""
    monkeypatch.setenv("FA2_SPLIT", "always")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("shape", [(8, 20, 300, 457), (2, 3, 640, 1000), (1, 4, 129, 1), (3, 5, 130, 190),
                                   (1, 1, 1000, 4096)])
def test_split_schedule_matches_oracle(D, shape, split_always):
    """Non-causal with a workspace: key-tile ranges cut across SMs, cut query tiles
    computed in parts and merged; every element against the oracle."""
    B, H, Lq, Lk = shape
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=1500 + D + Lq)
    o, lse, ws = run_ws(q, k, v, False, scale_of(D))
    o_ref, lse_ref = oracle.attention(q, k, v, False, scale_of(D))
    compare(o, lse, o_ref, lse_ref)
    # the arrival counters at the start of the workspace are zero again
    assert torch.count_nonzero(ws[:256]) == 0


@pytest.mark.parametrize("D", [64, 128, 256])
def test_split_schedule_deterministic_and_reusable(D, split_always):
    """Same inputs and workspace twice -> bit-identical output; causal ignores the workspace."""
    q, k, v = make_qkv(4, 8, 500, 700, D, seed_base=1600 + D)
    a = run_ws(q, k, v, False, scale_of(D))
    b = run_ws(q, k, v, False, scale_of(D), ws=a[2])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c_ws = run_ws(q, k, v, True, scale_of(D), ws=a[2])
    c_plain = run_cuda(q, k, v, True, scale_of(D))
    assert torch.equal(c_ws[0], c_plain[0]) and torch.equal(c_ws[1], c_plain[1])


def test_split_cost_model(monkeypatch):
    """The default estimate takes the cut ranges for one long head (4 query tiles on
    152+ SMs) and not for many short heads (256 units of 8 key tiles);
    FA2_SPLIT=never/always override it."""
    from io_aware_exact_fa2_gb300 import fa2_workspace_size
    monkeypatch.delenv("FA2_SPLIT", raising=False)
    assert fa2_workspace_size(1, 1, 1000, 4096, 128, False) > 0
    assert fa2_workspace_size(4, 16, 1024, 1024, 128, False) == 0
    assert fa2_workspace_size(1, 1, 1000, 4096, 128, True) == 0
    monkeypatch.setenv("FA2_SPLIT", "never")
    assert fa2_workspace_size(1, 1, 1000, 4096, 128, False) == 0
    monkeypatch.setenv("FA2_SPLIT", "always")
    assert fa2_workspace_size(4, 16, 1024, 1024, 128, False) > 0
    assert fa2_workspace_size(4, 16, 1024, 1024, 128, True) == 0


def test_lq_zero_is_a_noop():
    """Lq == 0: FA2_OK and nothing is written."""
    from io_aware_exact_fa2_gb300 import _binding
    dev = torch.device("cuda:0")
    k = torch.zeros(1, 2, 5, 64, dtype=torch.bfloat16, device=dev)
    buf = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    lbuf = torch.zeros(16, dtype=torch.float32, device=dev)
    st = _binding._lib.fa2_fwd(buf.data_ptr(), k.data_ptr(), k.data_ptr(), buf.data_ptr(), lbuf.data_ptr(),
                               1, 2, 0, 5, 64, 0, 0.125, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(buf) == 0 and torch.count_nonzero(lbuf) == 0


@pytest.mark.parametrize("D", [64, 128, 256])
def test_outputs_stay_in_bounds(D):
    """Canaries before and after O and LSE stay untouched (rows >= Lq are never written)."""
    from io_aware_exact_fa2_gb300 import _binding
    B, H, Lq, Lk = 1, 2, 200, 300
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=700 + D)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    n_o, n_l, pad = B * H * Lq * D, B * H * Lq, 4096
    o_buf = torch.full((pad + n_o + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad + n_l + pad,), 7.0, dtype=torch.float32, device=dev)
    o = o_buf[pad:pad + n_o].view(B, H, Lq, D)
    lse = l_buf[pad:pad + n_l].view(B, H, Lq)
    _binding.fa2_fwd(qd, kd, vd, o, lse, True, scale_of(D))
    st, code = _binding.fa2_get_device_error()
    assert st == 0, code
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[pad + n_o:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[pad + n_l:] == 7.0)
    o_ref, lse_ref = oracle.attention(q, k, v, True, scale_of(D))
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_deterministic(D):
    """Same inputs twice -> bit-identical O and LSE (no atomics, fixed reduction order)."""
    q, k, v = make_qkv(2, 4, 777, 999, D, seed_base=800 + D)
    a = run_cuda(q, k, v, False, scale_of(D))
    b = run_cuda(q, k, v, False, scale_of(D))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_side_stream_and_inputs_untouched():
    q, k, v = make_qkv(1, 4, 384, 384, 128, seed_base=900)
    s = torch.cuda.Stream()
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_get_device_error
    o = torch.empty(1, 4, 384, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 4, 384, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        fa2_fwd(qd, kd, vd, o, lse, True, scale_of(128))
    st, code = fa2_get_device_error(s)
    assert st == 0, code
    assert torch.equal(qd.cpu(), q) and torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    o_ref, lse_ref = oracle.attention(q, k, v, True, scale_of(128))
    compare(o.cpu(), lse.cpu(), o_ref, lse_ref)


def test_from_host_entry_point():
    """Host buffers in and out through the C ABI (one chunk: copies, kernel, copies)."""
    from io_aware_exact_fa2_gb300 import fa2_fwd_from_host
    B, H, Lq, Lk, D = 2, 3, 250, 333, 128
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed_base=950)
    dev = torch.device("cuda:0")
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty(B, H, Lq, D, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(B, H, Lq, dtype=torch.float32).pin_memory()
    qd = torch.empty_like(q, device=dev)
    kd = torch.empty_like(k, device=dev)
    vd = torch.empty_like(v, device=dev)
    od = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=dev)
    ld = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
    fa2_fwd_from_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, False, scale_of(D))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(q, k, v, False, scale_of(D))
    compare(oh, lh, o_ref, lse_ref)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_from_host_chunked_back_to_back(causal):
    """Inputs large enough to be cut into several chunks of heads (15 heads, not a
    multiple of the chunk count), two calls in a row on a side stream that reuse the
    same device staging buffers with different inputs: the second call's copies must
    wait for the first call's kernels, and the stream must wait for both."""
    from io_aware_exact_fa2_gb300 import fa2_fwd_from_host
    B, H, Lq, Lk, D = 3, 5, 1000, 1500, 128
    dev = torch.device("cuda:0")
    inputs = [make_qkv(B, H, Lq, Lk, D, seed_base=970 + 10 * s) for s in range(2)]
    staging = [torch.empty(B, H, L, D, dtype=torch.bfloat16, device=dev) for L in (Lq, Lk, Lk)]
    od = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=dev)
    ld = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
    outs = [(torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16).pin_memory(),
             torch.full((B, H, Lq), float("nan"), dtype=torch.float32).pin_memory()) for _ in inputs]
    pinned = [tuple(t.pin_memory() for t in qkv) for qkv in inputs]
    side = torch.cuda.Stream(dev)
    for (qh, kh, vh), (oh, lh) in zip(pinned, outs):
        fa2_fwd_from_host(qh, kh, vh, oh, lh, *staging, od, ld, causal, scale_of(D), stream=side)
    side.synchronize()
    for (q, k, v), (oh, lh) in zip(inputs, outs):
        rows = sample_rows(B, H, Lq, n_random=256, seed=971)
        o_ref, lse_ref = oracle.attention_rows(q, k, v, causal, scale_of(D), rows)
        idx = torch.from_numpy(rows)
        compare(oh.reshape(-1, D)[idx], lh.reshape(-1)[idx], o_ref, lse_ref)
        assert torch.isfinite(oh.float()).all() and torch.isfinite(lh).all()


def test_causal_row0_is_v0_exactly():
    """Causal row 0 sees only key 0: P = 1 exactly, so O_0 = V_0 bit for bit."""
    q, k, v = make_qkv(2, 4, 256, 256, 128, seed_base=960)
    o, _ = run_cuda(q, k, v, True, scale_of(128))
    assert torch.equal(o[:, :, 0], v[:, :, 0])


def test_no_device_error_after_suite():
    from io_aware_exact_fa2_gb300 import fa2_get_device_error
    assert fa2_get_device_error() == (0, 0)
