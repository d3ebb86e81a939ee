"""The benchmark's own arithmetic, on the CPU: the algorithmic work it divides
by, the launch count it claims, which kernel it names dominant and against
which peak, and when it reports DRAM traffic from a committed capture."""
import hashlib
import os

import numpy as np
import pytest

import bench
from sparse_moe_transformer_selected_b300 import inputs as gen

PEAKS = {"hbm_gbs": 6486.1, "bf16_tflops": 1775.2, "bf16_tflops_sustained": 1407.0}


def test_mxfp4_bytes_per_expert_follow_the_format():
    """gpt-oss expert at d = W = 2880: each of the 2W·d + d·W weights is half a
    byte of E2M1 code plus 1/32 of an E8M0 scale byte, and the biases are bf16."""
    wl = gen.WORKLOADS["gptoss20b_decode"]
    counts = np.zeros(wl.E, dtype=np.int64)
    counts[:31] = 1
    w = bench.stage_work(wl, counts)
    n_gu, n_dn = 2 * 2880 * 2880, 2880 * 2880
    per_expert = n_gu // 2 + n_gu // 32 + 2 * 2880 * 2 + n_dn // 2 + n_dn // 32 + 2880 * 2
    assert per_expert == 13_236_480
    assert w["_active"] == 31
    # the fused kernel reads the active experts once, the two x term tables
    # once, and writes out once
    assert w["experts"]["bytes"] == 31 * per_expert + 32 * 2880 * 2 + 32 * 2880 * 2
    assert w["experts"]["flops"] == 2 * 128 * (2880 * 5760 + 2880 * 2880) + 2 * 128 * 2880


def test_prefill_gate_up_flops():
    wl = gen.WORKLOADS["gptoss20b_prefill"]
    w = bench.stage_work(wl, np.ones(wl.E, dtype=np.int64))
    assert w["gate_up"]["flops"] == 2 * 32768 * 2880 * 5760


@pytest.mark.parametrize("T,d,E,mx,want", [
    (32, 2880, 32, True, 3),      # logits, top-k with the scan, the fused expert kernel
    (200, 256, 8, False, 5),      # + the gather, gate_up and down as two kernels
    (300, 96, 8, False, 6),       # > 8 router tiles: the scan on its own; d % 64: no split
    (8192, 2880, 32, False, 7),   # ... and the router-weight split for the tensor-core logits
])
def test_launch_count_per_step(T, d, E, mx, want):
    assert bench.kernels_per_step(T, d, E, mx) == want


def test_roofline_names_the_dominant_kernel_and_its_peak():
    wl = gen.WORKLOADS["gptoss20b_prefill"]
    counts = np.full(wl.E, 1024, dtype=np.int64)
    stage_ms = {"router_topk": 0.04, "route_scan": 0.01, "route_scatter": 0.04,
                "gate_up": 1.0, "down_combine": 0.8}
    mma = {"f16_tmem_a_n128": 2304.0}
    roof, active = bench.roofline(wl, counts, stage_ms, 1.9, False, PEAKS, "measured", mma)
    assert active == 32 and roof["kernel"] == "gate_up" and roof["bound"] == "tensor"
    flops = 2 * 32768 * 2880 * 5760
    assert roof["achieved"] == pytest.approx(flops / 1e-3 / 1e12)
    # a step far under a second is timed against the burst peak
    assert roof["peak"] == PEAKS["bf16_tflops"]
    assert roof["frac"] == pytest.approx(roof["achieved"] / PEAKS["bf16_tflops"])
    assert roof["frac_of_form_peak"] == pytest.approx(roof["achieved"] / 2304.0)
    # down issues two MMAs per K step (h hi and lo)
    stage_ms["down_combine"] = 2.0
    roof, _ = bench.roofline(wl, counts, stage_ms, 3.1, False, PEAKS, "measured", mma)
    assert roof["kernel"] == "down_combine"
    assert roof["frac_of_form_peak"] == pytest.approx(2 * roof["achieved"] / 2304.0)


def test_roofline_of_a_decode_step_is_hbm_bound():
    wl = gen.WORKLOADS["gptoss20b_decode"]
    counts = np.zeros(wl.E, dtype=np.int64)
    counts[:31] = 4
    roof, _ = bench.roofline(wl, counts, {"router_topk": 0.0126, "experts": 0.0878}, 0.104,
                             True, PEAKS, "measured")
    assert roof["kernel"] == "experts" and roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(roof["algorithmic"]["bytes"] / 87.8e-6 / 1e9)
    assert roof["frac_of_8tbs"] == pytest.approx(roof["achieved"] / 8000.0)


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    csrc = tmp_path / "sparse_moe_transformer_selected_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "expert_gemm_mx.cu"
    src.write_bytes(b"// one version of a kernel\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# kernel workload sha bytes\n"
        f"experts gptoss20b_decode {sha} 418131968\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("experts", "gptoss20b_decode", True) == 418131968.0
    assert bench.kernel_traffic("experts", "gptoss120b_skew64", True) is None
    src.write_bytes(b"// the kernel changed since the capture\n")
    assert bench.kernel_traffic("experts", "gptoss20b_decode", True) is None


def test_committed_traffic_lines_use_the_benchmark_names():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    for line in open(path):
        p = line.split()
        if len(p) == 4 and not line.startswith("#"):
            assert p[0] in ("experts", "gate_up", "down_combine")   # the benchmark's stage names
            assert p[1] in gen.WORKLOADS
            assert len(p[2]) == 16 and int(p[3]) > 0
