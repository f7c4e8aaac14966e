"""fa2_fwd_noalloc: the split-schedule pass with its workspace taken from the
library's fixed per-device scratch instead of the caller.

The GPU tests compare it, bit for bit, with the existing workspace entry point
(fa2_fwd_ws with a workspace from fa2_workspace) on two calls in a row with
different inputs, so a scratch left dirty by one call would show in the next.
The file is named to be collected last; it also passes when run alone (the
first call then does the scratch set-up)."""
import ctypes
import os
import re

import pytest
import torch

from io_aware_exact_fa2_gb300 import build as fa2_build
from io_aware_exact_fa2_gb300.workloads import make_qkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def binding():
    fa2_build.build()
    from io_aware_exact_fa2_gb300 import _binding
    return _binding


def test_scratch_limit_matches_header(binding):
    text = open(os.path.join(ROOT, "include", "fa2.h")).read()
    m = re.search(r"#define\s+FA2_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "FA2_NOALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == binding.NOALLOC_SCRATCH_BYTES == 48 << 20


def test_noalloc_rejects_bad_arguments_on_the_host(binding):
    """Same host-side validation as fa2_fwd; no CUDA call is made for these."""
    lib = binding._lib
    P = 0x10000
    INVALID, UNSUPPORTED = 1, 2
    f = lib.fa2_fwd_noalloc
    assert f(0, P, P, P, P, 1, 1, 8, 8, 64, 0, 0.125, None) == INVALID
    assert f(P, P, P, P + 8, P, 1, 1, 8, 8, 64, 0, 0.125, None) == INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 0, 64, 0, 0.125, None) == INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 8, 64, 0, float("nan"), None) == INVALID
    assert f(P, P, P, P, P, 1, 1, 8, 8, 96, 0, 0.125, None) == UNSUPPORTED
    assert f(P, P, P, P, P, 1, 1, 0, 8, 64, 0, 0.125, None) == 0   # Lq == 0: no-op


# (B, H, Lq, Lk, D, causal, uses_scratch): the cut-range schedule for each D (it
# takes the scratch), one non-causal shape whose whole query tiles already fill the
# 152 SMs evenly (152 units of 8 key tiles: the cost model keeps whole units, no
# scratch), and a causal pass (never cut, no scratch)
CASES = [
    (1, 1, 1000, 4096, 128, False, True),
    (1, 1, 1000, 4096, 64, False, True),
    (1, 2, 700, 3000, 256, False, True),
    (2, 16, 4096, 4096, 128, False, True),
    (2, 3, 640, 1000, 128, False, True),
    (2, 76, 256, 1024, 64, False, False),
    (1, 2, 900, 900, 128, True, False),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dH%dLq%dLk%dD%d%s" % (c[:5] + ("c" if c[5] else "",)))
def test_noalloc_matches_workspace_entry_point_twice(binding, case):
    B, H, Lq, Lk, D, causal, uses_scratch = case
    dev = torch.device("cuda:0")
    scale = D ** -0.5
    inputs = [tuple(t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed_base=7000 + 10 * D + s))
              for s in range(2)]
    refs = []
    for q, k, v in inputs:
        o = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
        binding.fa2_fwd(q, k, v, o, lse, causal, scale, workspace=binding.fa2_workspace(q, k, causal))
        refs.append((o, lse))
    need = binding.fa2_workspace_size(B, H, Lq, Lk, D, causal)
    assert need <= binding.NOALLOC_SCRATCH_BYTES
    # the case takes the path it is meant to cover: cut ranges through the scratch,
    # or whole query tiles without it
    assert (need > 0) == uses_scratch, need

    outs = [(torch.full((B, H, Lq, D), float("nan"), dtype=torch.bfloat16, device=dev),
             torch.full((B, H, Lq), float("nan"), dtype=torch.float32, device=dev)) for _ in inputs]
    torch.cuda.synchronize()
    free_before = None
    for i, ((q, k, v), (o, lse)) in enumerate(zip(inputs, outs)):
        binding.fa2_fwd_noalloc(q, k, v, o, lse, causal, scale)
        torch.cuda.synchronize()
        if i == 0:
            free_before = torch.cuda.mem_get_info(dev)[0]
    # the second call allocated nothing on the device
    assert torch.cuda.mem_get_info(dev)[0] == free_before
    st, code = binding.fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    for (o, lse), (o_ref, lse_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


@pytest.mark.gpu
def test_noalloc_back_to_back_on_one_stream(binding):
    """Two calls enqueued back to back without a host sync in between (ordered on
    one stream, so they share the scratch safely) match the workspace entry point."""
    B, H, Lq, Lk, D = 1, 1, 1000, 4096, 128
    dev = torch.device("cuda:0")
    assert binding.fa2_workspace_size(B, H, Lq, Lk, D, False) > 0   # the cut-range path
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed_base=7500))
    o_ref = torch.empty(B, H, Lq, D, dtype=torch.bfloat16, device=dev)
    lse_ref = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
    binding.fa2_fwd(q, k, v, o_ref, lse_ref, False, workspace=binding.fa2_workspace(q, k, False))
    o1, o2 = torch.empty_like(o_ref), torch.empty_like(o_ref)
    l1, l2 = torch.empty_like(lse_ref), torch.empty_like(lse_ref)
    binding.fa2_fwd_noalloc(q, k, v, o1, l1, False)
    binding.fa2_fwd_noalloc(q, k, v, o2, l2, False)
    st, code = binding.fa2_get_device_error()
    assert st == 0, f"device error {code:#x}"
    assert torch.equal(o1, o_ref) and torch.equal(o2, o_ref)
    assert torch.equal(l1, lse_ref) and torch.equal(l2, lse_ref)
