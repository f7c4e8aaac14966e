"""The forward kernel's bounded waits: a wait between warps that runs out is
reported by fa2_get_device_error as FA2_ERR_TIMEOUT, the kernel winds down
without hanging, and the next call on the same context is clean.

The time-out is made on purpose with the library's test switch FA2_TEST_STALL=1:
the softmax warps first wait on a barrier that nothing completes.  That wait
runs out after FA2_TEST_WAIT_LIMIT_NS (200 us here), the softmax warps leave, and
the MMA warp's and producer's waits on them run out in turn.  Nothing faults:
before exiting, each CTA still waits, with the full one-second bound, for the TMA
copies and MMAs it has already issued (the producer for its loads, the MMA warp
for its MMAs through a final commit), and only then frees its tensor memory.
"""
import pytest
import torch

import oracle
from io_aware_exact_fa2_gb300.workloads import WORKLOADS, workload_inputs
from parity import compare, run_cuda

pytestmark = pytest.mark.gpu

FA2_ERR_TIMEOUT = 4


def test_inter_warp_time_out_is_reported_and_the_next_call_is_clean(monkeypatch):
    from io_aware_exact_fa2_gb300 import fa2_fwd, fa2_get_device_error
    w = WORKLOADS["c1"]
    q, k, v = workload_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    assert fa2_get_device_error() == (0, 0)   # nothing pending from earlier tests

    monkeypatch.setenv("FA2_TEST_STALL", "1")
    monkeypatch.setenv("FA2_TEST_WAIT_LIMIT_NS", "200000")
    fa2_fwd(qd, kd, vd, o, lse, False, w.scale)
    st, code = fa2_get_device_error()
    assert st == FA2_ERR_TIMEOUT, (st, hex(code))
    # a wait between warps ran out (producer 1, MMA 2, softmax 3; the stalled softmax
    # wait is 0x30f); never a CTA's own drain of its copies and MMAs (4), which keeps
    # the full bound
    assert (code >> 8) in (1, 2, 3), hex(code)
    assert fa2_get_device_error() == (0, 0)   # read and cleared

    monkeypatch.delenv("FA2_TEST_STALL")
    monkeypatch.delenv("FA2_TEST_WAIT_LIMIT_NS")
    for causal in (False, True):
        o2, lse2 = run_cuda(q, k, v, causal, w.scale)   # asserts a clean error word
        o_ref, lse_ref = oracle.attention(q, k, v, causal, w.scale)
        compare(o2, lse2, o_ref, lse_ref)
