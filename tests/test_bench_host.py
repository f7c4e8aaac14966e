"""Host-side logic of bench.py, on the CPU: the metric's FLOP and byte counts,
clock-sample parsing, the traffic record's staleness check, the reference arm,
and the multi-process (torchrun-style) timing reduction over gloo ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from io_aware_exact_fa2_gb300.workloads import WORKLOADS  # noqa: E402


def test_window_flops_count_visible_pairs():
    """Sliding window: 4*D FLOPs per visible pair, query i seeing keys max(0, i - w) .. i;
    checked against a direct count, and w >= Lq - 1 equals the causal count plus the diagonal."""
    class W:
        B, H, D = 2, 3, 64
    for lq, win in [(1, 0), (5, 0), (5, 2), (5, 4), (5, 10), (300, 100), (129, 128)]:
        W.Lq = lq
        direct = sum(min(i, win) + 1 for i in range(lq))
        assert bench.window_flops(W, win) == 4 * W.B * W.H * W.D * direct
    c4 = WORKLOADS["c4"]
    full = bench.window_flops(c4, c4.Lq)
    assert full == 4 * c4.B * c4.H * c4.D * c4.Lq * (c4.Lq + 1) // 2
    assert full - c4.flops(True) == 4 * c4.B * c4.H * c4.D * c4.Lq / 2


def test_flop_and_byte_counts():
    """FLOPs = 4*B*H*Lq*Lk*D (halved for causal); bytes = Q,K,V read once + O, LSE written once."""
    c3 = WORKLOADS["c3"]
    assert c3.flops(False) == 4 * 2 * 16 * 4096 * 4096 * 128 == 274877906944
    assert c3.flops(True) == c3.flops(False) / 2
    assert c3.algorithmic_bytes() == 2 * 16 * (2 * 4096 * 128 * 2 + 2 * 4096 * 128 * 2 + 4 * 4096)
    c5 = WORKLOADS["c5"]
    assert c5.flops(False) == 4 * 2 * 8 * 2000 * 3000 * 256
    assert c5.peaky_every == 64 and c5.modes == ("noncausal",)


def test_clock_summary():
    line = "2026/12/02 08:00:00.000, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {cap}"
    lines = [(10.0, line.format(mhz=2070, cap="Not Active")),
             (10.1, line.format(mhz=1980, cap="Active")),
             (10.2, line.format(mhz=2010, cap="Not Active")),
             (20.0, line.format(mhz=500, cap="Not Active"))]   # outside the region
    s = bench.ClockSampler.summarize(lines, 10.0, 10.2)
    assert s["samples"] == 3 and s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 900.5


def test_traffic_record_tracks_kernel_source(tmp_path, monkeypatch):
    from io_aware_exact_fa2_gb300 import build as fa2_build
    digest = fa2_build.kernel_digest()
    rec = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if os.path.exists(rec):
        d = json.load(open(rec))
        for name in d.get("workloads", {}):
            got = bench.load_traffic(digest, name)
            assert (got is not None) == (d["kernel_source_digest"] == digest)
            if got is not None:
                assert got["dram_bytes_per_launch"] > 0
    assert bench.load_traffic("not-a-digest", "c4") is None


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c1", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # each rank reports its own elapsed time; every rank must see the max
    m = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    out[rank] = m
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}
